// ln_bwd.cu -- backward kernels of the fused residual-add + LayerNorm.
//
// Row gradient, HW4 form ("Accelerating Transformer on GPU (II): Training with LightSeq2",
// section 2.1), with the two row sums reduced together (section 2.2):
//   xhat = (s - mu) * rstd,  g = gamma * dy,
//   dx = rstd * (g - (sum g + xhat * sum g xhat) / n).
// Column gradients (sections 2.1 and 2.4): dgamma = sum_rows dy * xhat, dbeta = sum_rows dy.
//
// g = gamma * dy is rounded once (__fmul_rn, never fused into a later subtraction) so that
// the g in the row sums and the g in dx are the same number: when rstd is large (a row of
// near-constant values) any difference between them would be amplified into dx.
//
// Column sums, deterministic and without float atomics, in two stages:
//  1. Each block owns a FIXED contiguous range of rows.  While it computes dx it
//     accumulates dy * xhat and dy for the columns its threads own and, at the end, writes
//     one row of partial sums per statistic to the workspace: part[stat][block][col].
//  2. Every block then takes a ticket from an integer counter (atomicAdd).  The blocks whose
//     tickets are among the last F are the finishers: each waits (bounded) until all blocks
//     have arrived, then sums the partials of ITS slice of columns over blocks in a fixed
//     order and writes dgamma and dbeta.  The last finisher puts the counters back to 0.
//  This is the last-block-finishes idea of llm.c's layernorm_backward_kernel10 ("llm.c: the
//  llmc/ CUDA kernel layer", section 3.3), widened from one finishing block to F so that
//  the finish is spread over many SMs instead of serialising one SM on all partials.  The
//  grid is launched cooperatively, so every block is resident and the wait always ends.
//  Which block adds which rows, and in what order, depends only on (rows, cols, device),
//  so dgamma and dbeta are bitwise reproducible run to run.
//
// Accuracy of the column sums.  A plain fp32 sum of n terms of size sigma carries an error
// of about 2^-24 * sigma * sqrt(n * L) for chains of L additions, whatever the order: for
// 262144 rows that is ~1e-4, far above the 2e-5 that fp32 results are held to.  So:
//  * the block kernels keep each thread's running sums compensated (Kahan: a second fp32
//    register holds the rounding error of every addition) whenever a thread owns at most 16
//    columns (rows up to 8192 columns wide; wider rows keep plain fp32 sums: the registers
//    for compensation are not there);
//  * the warp (tile) kernel (bf16, short per-lane chains) keeps plain per-lane sums and
//    combines its warps with error-free additions (TwoSum);
//  * partial sums are stored as (hi, lo) fp32 pairs and the finishers add them with TwoSum,
//    so the only rounding left at the end is the final one to the output type.
#include <algorithm>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

// Consumer warps = rows per tile, plus one producer warp: 8 warps, because registers are
// allocated to warps in groups of four (a 9-warp block would pay for 12).
constexpr int kTileRows = 7;
constexpr int kTileThreads = (kTileRows + 1) * 32;
constexpr int kBwdBlockMaxThreads = 512;
constexpr int kBwdScalarThreads = 256;
constexpr int kMaxStages = 4;
// The warp kernel is used for bf16 rows of up to 5 vectors per lane (1280 columns) and at
// most this many rows, which keeps its plain per-lane chains short.
constexpr int kWarpPathMaxRows = 65536;

struct KParams {
    const void* dy;
    const void* xr;
    const void* gamma;
    const float* mean;
    const float* rstd;
    void* dx;
    void* dgamma;
    void* dbeta;
    int rows;
    int cols;
    float2* part;  // [2][gridDim.x][cols] (hi, lo) pairs
    unsigned* ctr;
    unsigned* status;
    uint64_t limit_ns;
    unsigned wait_extra;
    int finishers;
    int stages;
};

__device__ __forceinline__ void row_range(int rows, int& r0, int& r1) {
    r0 = (int)((long long)blockIdx.x * rows / gridDim.x);
    r1 = (int)((long long)(blockIdx.x + 1) * rows / gridDim.x);
}

// (S, C) += (h, l), where a compensated value is S + C.
__device__ __forceinline__ void comp_add(float& S, float& C, float h, float l) {
    float s, e;
    two_sum_f(S, h, s, e);
    S = s;
    C += e + l;
}

// Kahan step: the running value is s - c.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

// ---------------------------------------------------------------------------------------
// Stage 2: the finishers.  Finisher f of F owns the column groups [g0, g1) (a group is U
// adjacent columns).  Threads are arranged as Q subsets of the blocks times the (stat,
// group) units of the slice; thread (q, u) adds the (hi, lo) partials of blocks q, q+Q,
// q+2Q, ... in increasing order, then the Q subtotals of each unit are added in q order.
// `scratch` is shared memory of at least blockDim.x * 4 floats.
// ---------------------------------------------------------------------------------------
template <typename T, int U>
__device__ void finish_slice(const KParams& a, int P, int F, int f, float* scratch) {
    using IO = Io<T>;
    const int cols = a.cols;
    const int threads = blockDim.x;
    const int ngroups = cols / U;
    const int g0 = (int)((long long)f * ngroups / F);
    const int g1 = (int)((long long)(f + 1) * ngroups / F);
    const int wg = g1 - g0;
    const int units = 2 * wg;
    if (units == 0) return;
    T* dst[2] = {static_cast<T*>(a.dgamma), static_cast<T*>(a.dbeta)};
    const size_t stat_stride = (size_t)P * cols;
    const int tid = threadIdx.x;

    auto add_group = [&](float (&S)[U], float (&C)[U], const float2* src) {
        if constexpr (U == 2) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
            comp_add(S[0], C[0], v.x, v.y);
            comp_add(S[1], C[1], v.z, v.w);
        } else {
            const float2 v = __ldcg(src);
            comp_add(S[0], C[0], v.x, v.y);
        }
    };
    auto store = [&](int u, const float (&S)[U], const float (&C)[U]) {
        const int stat = u / wg, grp = g0 + u % wg;
#pragma unroll
        for (int i = 0; i < U; ++i) dst[stat][(size_t)grp * U + i] = IO::from_f(S[i] + C[i]);
    };

    if (units >= threads) {
        for (int u = tid; u < units; u += threads) {
            const int stat = u / wg, grp = g0 + u % wg;
            const float2* src = a.part + stat * stat_stride + (size_t)grp * U;
            float S[U], C[U];
#pragma unroll
            for (int i = 0; i < U; ++i) S[i] = C[i] = 0.f;
#pragma unroll 8
            for (int p = 0; p < P; ++p) add_group(S, C, src + (size_t)p * cols);
            store(u, S, C);
        }
        return;
    }
    const int Q = threads / units;
    const int q = tid / units, u = tid % units;
    if (q < Q) {
        const int stat = u / wg, grp = g0 + u % wg;
        const float2* src = a.part + stat * stat_stride + (size_t)grp * U;
        float S[U], C[U];
#pragma unroll
        for (int i = 0; i < U; ++i) S[i] = C[i] = 0.f;
#pragma unroll 8
        for (int p = q; p < P; p += Q) add_group(S, C, src + (size_t)p * cols);
        float* sc = scratch + ((size_t)q * units + u) * (2 * U);
#pragma unroll
        for (int i = 0; i < U; ++i) {
            sc[2 * i] = S[i];
            sc[2 * i + 1] = C[i];
        }
    }
    __syncthreads();
    for (int v = tid; v < units; v += threads) {
        float S[U], C[U];
#pragma unroll
        for (int i = 0; i < U; ++i) S[i] = C[i] = 0.f;
        for (int qq = 0; qq < Q; ++qq) {
            const float* sc = scratch + ((size_t)qq * units + v) * (2 * U);
#pragma unroll
            for (int i = 0; i < U; ++i) comp_add(S[i], C[i], sc[2 * i], sc[2 * i + 1]);
        }
        store(v, S, C);
    }
}

// Called by every thread of every block after its partial row is written.
template <typename T>
__device__ void arrive_and_finish(const KParams& a, float* scratch) {
    __shared__ unsigned s_ticket;
    __shared__ int s_ok;
    __threadfence();  // this thread's partial sums are visible GPU-wide before the ticket
    __syncthreads();
    const unsigned P = gridDim.x;
    const unsigned F = (unsigned)a.finishers;
    if (threadIdx.x == 0) s_ticket = atomicAdd(&a.ctr[0], 1u);
    __syncthreads();
    const unsigned ticket = s_ticket;
    if (ticket < P - F) return;  // not among the last F arrivals: done
    const int f = (int)(ticket - (P - F));
    if (threadIdx.x == 0) {
        const bool ok = wait_counter_geq(&a.ctr[0], P + a.wait_extra, a.limit_ns);
        __threadfence();
        s_ok = ok ? 1 : 0;
        if (!ok) raise_status(a.status, kStatusTimeout);
    }
    __syncthreads();
    if (!s_ok) return;
    if (a.cols % 2 == 0)
        finish_slice<T, 2>(a, (int)P, (int)F, f, scratch);
    else
        finish_slice<T, 1>(a, (int)P, (int)F, f, scratch);
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(&a.ctr[1], 1u);
        if (done == F - 1) {  // every finisher is past its wait: reset for the next call
            atomicExch(&a.ctr[0], 0u);
            atomicExch(&a.ctr[1], 0u);
        }
    }
}

// ---------------------------------------------------------------------------------------
// Warp per row, fed by a bulk-copy (TMA) pipeline (the forward's tile kernel, for dy and x).
// The block owns a fixed contiguous range of tiles (7 consecutive rows each); the producer
// warp's lane 0 fetches each tile of dy and of x with one cp.async.bulk apiece, `stages`
// tiles ahead; consumer warp w handles row w of every tile.  Lane l owns the columns of
// vectors l, l+32, ... in every row, so its column sums stay in registers; at the end the
// 7 consumer warps' sums are added in warp order with TwoSum through shared memory (the
// drained ring), one statistic at a time, into the block's (hi, lo) partial row.
// ---------------------------------------------------------------------------------------
template <typename T, int VPL>
__global__ void __launch_bounds__(kTileThreads, VPL <= 3 ? 2 : 1) bwd_tile_kernel(const KParams a) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = a.cols, nvec = cols / V, stages = a.stages, rows = a.rows;
    const float fcols = (float)cols;
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned tile_bytes = (unsigned)kTileRows * row_bytes;
    const unsigned slot_bytes = 2u * tile_bytes;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    int t0, t1;
    row_range((rows + kTileRows - 1) / kTileRows, t0, t1);  // this block's tiles
    const int my_tiles = t1 - t0;

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kTileRows);
        }
        fence_barrier_init();
    }
    __syncthreads();

    float accg[VPL][V], accb[VPL][V];
#pragma unroll
    for (int v = 0; v < VPL; ++v)
#pragma unroll
        for (int k = 0; k < V; ++k) accg[v][k] = accb[v][k] = 0.f;

    if (warp == kTileRows) {  // producer
        if (lane == 0) {
            int k = 0;
            for (; k < my_tiles; ++k) {
                const int slot = k % stages;
                if (k >= stages &&
                    !mbar_wait(&empty_bar[slot], (unsigned)(k / stages - 1) & 1u, a.limit_ns)) {
                    raise_status(a.status, kStatusTimeout);
                    break;
                }
                const int r0 = (t0 + k) * kTileRows;
                const unsigned bytes = (unsigned)min(kTileRows, rows - r0) * row_bytes;
                unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
                mbar_arrive_expect_tx(&full_bar[slot], 2u * bytes);
                bulk_g2s(dst, dy + (size_t)r0 * cols, bytes, &full_bar[slot]);
                bulk_g2s(dst + tile_bytes, xr + (size_t)r0 * cols, bytes, &full_bar[slot]);
            }
            for (int j = max(0, k - stages); j < k; ++j)  // drain: every copy has landed
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, a.limit_ns);
        }
    } else {  // consumers
        float gm[VPL][V];  // gamma of this lane's columns, unpacked once
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const int vi = v * 32 + lane;
            IO::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gm[v]);
        }
        // mean and rstd of the warp's row in the next tile are loaded one tile ahead, so
        // their latency is not on the row's critical path.
        int row = t0 * kTileRows + warp;
        float mu_next = row < rows ? a.mean[row] : 0.f;
        float rs_next = row < rows ? a.rstd[row] : 0.f;
        for (int k = 0; k < my_tiles; ++k, row += kTileRows) {
            const int slot = k % stages;
            const float mu = mu_next, rs = rs_next;
            if (row + kTileRows < rows && k + 1 < my_tiles) {
                mu_next = a.mean[row + kTileRows];
                rs_next = a.rstd[row + kTileRows];
            }
            const bool ok = mbar_wait(&full_bar[slot], (unsigned)(k / stages) & 1u, a.limit_ns);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) raise_status(a.status, kStatusTimeout);
                break;
            }
            if (row < rows) {
                const size_t base = (size_t)row * cols;
                const T* dys = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes +
                                                          (size_t)warp * row_bytes);
                const T* xs = dys + (size_t)kTileRows * cols;
                float sg0 = 0.f, sg1 = 0.f, sgx0 = 0.f, sgx1 = 0.f;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const int vi = v * 32 + lane;
                    if (vi < nvec) {
                        float d[V], xx[V];
                        IO::unpack(*reinterpret_cast<const uint4*>(dys + (size_t)vi * V), d);
                        IO::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)vi * V), xx);
#pragma unroll
                        for (int q = 0; q < V; q += 2) {
                            const float xh0 = (xx[q] - mu) * rs, xh1 = (xx[q + 1] - mu) * rs;
                            const float g0 = __fmul_rn(gm[v][q], d[q]);
                            const float g1 = __fmul_rn(gm[v][q + 1], d[q + 1]);
                            sg0 += g0;
                            sg1 += g1;
                            sgx0 = fmaf(g0, xh0, sgx0);
                            sgx1 = fmaf(g1, xh1, sgx1);
                            accg[v][q] = fmaf(d[q], xh0, accg[v][q]);
                            accg[v][q + 1] = fmaf(d[q + 1], xh1, accg[v][q + 1]);
                            accb[v][q] += d[q];
                            accb[v][q + 1] += d[q + 1];
                        }
                    }
                }
                float sg = sg0 + sg1, sgx = sgx0 + sgx1;
                warp_sum2(sg, sgx);  // the one reduction of the row: both sums together
                // dx = rs * (g - (mg + xhat * mgx)) with the same rounded g as in the sums, so
                // g - mg cancels exactly where it should (a one-column row gives dx = 0).
                const float mg = sg / fcols, mgx = sgx / fcols;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const int vi = v * 32 + lane;
                    if (vi < nvec) {  // second pass re-reads the row from shared memory
                        float d[V], xx[V], o[V];
                        IO::unpack(*reinterpret_cast<const uint4*>(dys + (size_t)vi * V), d);
                        IO::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)vi * V), xx);
#pragma unroll
                        for (int q = 0; q < V; ++q) {
                            const float xh = (xx[q] - mu) * rs;
                            o[q] = rs * (__fmul_rn(gm[v][q], d[q]) - fmaf(xh, mgx, mg));
                        }
                        st_stream(dx + base + (size_t)vi * V, IO::pack(o));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
        }
    }
    __syncthreads();  // the ring is drained and no warp reads it any more

    // Block partial row: add the consumer warps' sums in warp order (TwoSum), one statistic
    // at a time, and store the (hi, lo) pair.
    float* smem_f = reinterpret_cast<float*>(smem_raw);  // [kTileRows][cols]
    const int P = gridDim.x;
#pragma unroll
    for (int stat = 0; stat < 2; ++stat) {
        if (warp < kTileRows) {
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * 32 + lane;
                if (vi < nvec) {
                    float* dst = smem_f + (size_t)warp * cols + (size_t)vi * V;
#pragma unroll
                    for (int k = 0; k < V; k += 4)
                        *reinterpret_cast<float4*>(dst + k) =
                            stat == 0 ? make_float4(accg[v][k], accg[v][k + 1], accg[v][k + 2], accg[v][k + 3])
                                      : make_float4(accb[v][k], accb[v][k + 1], accb[v][k + 2], accb[v][k + 3]);
                }
            }
        }
        __syncthreads();
        float2* prow = a.part + ((size_t)stat * P + blockIdx.x) * cols;
        for (int c = tid; c < cols; c += blockDim.x) {
            float S = 0.f, C = 0.f;
#pragma unroll
            for (int w = 0; w < kTileRows; ++w) comp_add(S, C, smem_f[(size_t)w * cols + c], 0.f);
            prow[c] = make_float2(S, C);
        }
        __syncthreads();
    }
    arrive_and_finish<T>(a, smem_f);
}

// ---------------------------------------------------------------------------------------
// Block per row with bulk-copy staging of dy and x rows (several rows ahead).  Thread t of
// the block (blockDim.x threads) owns the columns of vectors t, t + blockDim.x, ... in
// every row, so its column sums stay in registers (compensated when KAHAN) and go straight
// to the block's partial row.
// ---------------------------------------------------------------------------------------
template <typename T, int VPT, bool KAHAN>
__global__ void __launch_bounds__(kBwdBlockMaxThreads, 1) bwd_block_kernel(const KParams a) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    constexpr int MAXW = kBwdBlockMaxThreads / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages];
    __shared__ float red[2][MAXW];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nw = nthreads >> 5;
    const int cols = a.cols, nvec = cols / V, stages = a.stages;
    const float fcols = (float)cols;
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned slot_bytes = 2u * row_bytes;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    int r0, r1;
    row_range(a.rows, r0, r1);

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&full_bar[i], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int k) {  // thread 0 only: fetch row r0 + k
        const int row = r0 + k;
        if (row >= r1) return;
        const int slot = k % stages;
        unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], slot_bytes);
        bulk_g2s(dst, dy + (size_t)row * cols, row_bytes, &full_bar[slot]);
        bulk_g2s(dst + row_bytes, xr + (size_t)row * cols, row_bytes, &full_bar[slot]);
    };
    if (tid == 0)
        for (int k = 0; k < stages; ++k) issue(k);

    uint4 gv[VPT];
    float sg_hi[VPT][V], sb_hi[VPT][V];  // running sums of dy * xhat and dy
    float sg_c[KAHAN ? VPT : 1][V], sb_c[KAHAN ? VPT : 1][V];  // Kahan compensations
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = v * nthreads + tid;
        gv[v] = vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < V; ++k) sg_hi[v][k] = sb_hi[v][k] = 0.f;
    }
#pragma unroll
    for (int v = 0; v < (KAHAN ? VPT : 1); ++v)
#pragma unroll
        for (int k = 0; k < V; ++k) sg_c[v][k] = sb_c[v][k] = 0.f;

    int k = 0;
    // mean and rstd are loaded one row ahead (off the row's critical path).
    float mu_next = r0 < r1 ? a.mean[r0] : 0.f, rs_next = r0 < r1 ? a.rstd[r0] : 0.f;
    for (int row = r0; row < r1; ++row, ++k) {
        const int slot = k % stages;
        const float mu = mu_next, rs = rs_next;
        if (row + 1 < r1) {
            mu_next = a.mean[row + 1];
            rs_next = a.rstd[row + 1];
        }
        if (!mbar_wait(&full_bar[slot], (unsigned)(k / stages) & 1u, a.limit_ns)) abort_flag = 1;
        const T* dys = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes);
        const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes + row_bytes);
        const size_t base = (size_t)row * cols;
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                float d[V], xx[V], gm[V];
                IO::unpack(*reinterpret_cast<const uint4*>(dys + (size_t)vi * V), d);
                IO::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)vi * V), xx);
                IO::unpack(gv[v], gm);
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    const float xh = (xx[q] - mu) * rs;
                    const float g = __fmul_rn(gm[q], d[q]);
                    sg += g;
                    sgx += g * xh;
                    if constexpr (KAHAN) {
                        kahan_add(sg_hi[v][q], sg_c[v][q], __fmul_rn(d[q], xh));
                        kahan_add(sb_hi[v][q], sb_c[v][q], d[q]);
                    } else {
                        sg_hi[v][q] += d[q] * xh;
                        sb_hi[v][q] += d[q];
                    }
                }
            }
        }
        warp_sum2(sg, sgx);
        if (lane == 0) {
            red[0][warp] = sg;
            red[1][warp] = sgx;
        }
        __syncthreads();  // the one cross-warp exchange of the row
        if (abort_flag) break;
        float tg = 0.f, tgx = 0.f;
        for (int w = 0; w < nw; ++w) {  // same order in every thread
            tg += red[0][w];
            tgx += red[1][w];
        }
        const float mg = tg / fcols, mgx = tgx / fcols;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                float d[V], xx[V], gm[V], o[V];
                IO::unpack(*reinterpret_cast<const uint4*>(dys + (size_t)vi * V), d);
                IO::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)vi * V), xx);
                IO::unpack(gv[v], gm);
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    const float xh = (xx[q] - mu) * rs;
                    o[q] = rs * (__fmul_rn(gm[q], d[q]) - (mg + xh * mgx));
                }
                st_stream(dx + base + (size_t)vi * V, IO::pack(o));
            }
        }
        __syncthreads();  // slot and `red` free again
        if (tid == 0) issue(k + stages);
    }

    if (abort_flag) {
        if (tid == 0) {
            raise_status(a.status, kStatusTimeout);
            for (int j = k; j < k + stages && r0 + j < r1; ++j)
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, a.limit_ns);
        }
        __syncthreads();
        return;  // no partial row: the finishers' bounded wait runs out as well
    }

    const int P = gridDim.x;
#pragma unroll
    for (int stat = 0; stat < 2; ++stat) {
        float2* prow = a.part + ((size_t)stat * P + blockIdx.x) * cols;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
#pragma unroll
                for (int q = 0; q < V; q += 2) {
                    float h0, h1, l0 = 0.f, l1 = 0.f;
                    h0 = stat == 0 ? sg_hi[v][q] : sb_hi[v][q];
                    h1 = stat == 0 ? sg_hi[v][q + 1] : sb_hi[v][q + 1];
                    if constexpr (KAHAN) {  // Kahan's value is s - c
                        l0 = -(stat == 0 ? sg_c[v][q] : sb_c[v][q]);
                        l1 = -(stat == 0 ? sg_c[v][q + 1] : sb_c[v][q + 1]);
                    }
                    *reinterpret_cast<float4*>(prow + (size_t)vi * V + q) =
                        make_float4(h0, l0, h1, l1);
                }
            }
        }
    }
    arrive_and_finish<T>(a, reinterpret_cast<float*>(smem_raw));
}

// ---------------------------------------------------------------------------------------
// Scalar kernel (any alignment, any width).  Each column is owned by one thread of the
// block; its compensated running sums live in shared memory when 16 bytes per column fit,
// else directly in the block's partial row of the workspace (L2-resident).
// ---------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kBwdScalarThreads) bwd_scalar_kernel(const KParams a) {
    using IO = Io<T>;
    constexpr int NW = kBwdScalarThreads / 32;
    extern __shared__ __align__(16) float smem_f[];
    __shared__ float red[2][NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = a.cols, P = gridDim.x;
    const float fcols = (float)cols;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    int r0, r1;
    row_range(a.rows, r0, r1);
    // acc_g[c] = (s, c) Kahan pair of dgamma, acc_b[c] the one of dbeta.
    const bool in_smem = a.stages != 0;  // the host sets it when 16 * cols bytes fit
    float2* acc_g = in_smem ? reinterpret_cast<float2*>(smem_f)
                            : a.part + (size_t)blockIdx.x * cols;
    float2* acc_b = in_smem ? reinterpret_cast<float2*>(smem_f) + cols
                            : a.part + ((size_t)P + blockIdx.x) * cols;
    for (int j = tid; j < cols; j += kBwdScalarThreads)
        acc_g[j] = acc_b[j] = make_float2(0.f, 0.f);

    for (int row = r0; row < r1; ++row) {
        const size_t base = (size_t)row * cols;
        const float mu = a.mean[row], rs = a.rstd[row];
        float sg = 0.f, sgx = 0.f;
        for (int j = tid; j < cols; j += kBwdScalarThreads) {
            const float d = IO::to_f(dy[base + j]);
            const float xh = (IO::to_f(xr[base + j]) - mu) * rs;
            const float g = __fmul_rn(IO::to_f(gamma[j]), d);
            sg += g;
            sgx += g * xh;
            float2 pg = acc_g[j], pb = acc_b[j];
            kahan_add(pg.x, pg.y, __fmul_rn(d, xh));
            kahan_add(pb.x, pb.y, d);
            acc_g[j] = pg;
            acc_b[j] = pb;
        }
        warp_sum2(sg, sgx);
        if (lane == 0) {
            red[0][warp] = sg;
            red[1][warp] = sgx;
        }
        __syncthreads();
        float tg = 0.f, tgx = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            tg += red[0][w];
            tgx += red[1][w];
        }
        const float mg = tg / fcols, mgx = tgx / fcols;
        for (int j = tid; j < cols; j += kBwdScalarThreads) {
            const float d = IO::to_f(dy[base + j]);
            const float xh = (IO::to_f(xr[base + j]) - mu) * rs;
            dx[base + j] = IO::from_f(rs * (__fmul_rn(IO::to_f(gamma[j]), d) - (mg + xh * mgx)));
        }
        __syncthreads();
    }
    // Partial row as (hi, lo): Kahan's value is s - c.
    for (int j = tid; j < cols; j += kBwdScalarThreads) {
        const float2 pg = acc_g[j], pb = acc_b[j];
        a.part[(size_t)blockIdx.x * cols + j] = make_float2(pg.x, -pg.y);
        a.part[((size_t)P + blockIdx.x) * cols + j] = make_float2(pb.x, -pb.y);
    }
    __syncthreads();  // the shared accumulators become the finish scratch
    arrive_and_finish<T>(a, smem_f);
}

// ---------------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------------
// Warp path: up to 8 vectors per lane for fp32 (1024 columns), 5 for bf16 (1280 columns):
// beyond that the register-resident column sums no longer fit without spilling.
template <typename T>
const void* warp_kernel(int vpl) {
    if constexpr (Io<T>::kVec == 8) {
        switch (vpl) {
            case 1: return (const void*)bwd_tile_kernel<T, 1>;
            case 2: return (const void*)bwd_tile_kernel<T, 2>;
            case 3: return (const void*)bwd_tile_kernel<T, 3>;
            case 4: return (const void*)bwd_tile_kernel<T, 4>;
            case 5: return (const void*)bwd_tile_kernel<T, 5>;
            default: return nullptr;
        }
    } else {
        switch (vpl) {
            case 1: return (const void*)bwd_tile_kernel<T, 1>;
            case 2: return (const void*)bwd_tile_kernel<T, 2>;
            case 3: return (const void*)bwd_tile_kernel<T, 3>;
            case 4: return (const void*)bwd_tile_kernel<T, 4>;
            case 5: return (const void*)bwd_tile_kernel<T, 5>;
            case 6: return (const void*)bwd_tile_kernel<T, 6>;
            case 7: return (const void*)bwd_tile_kernel<T, 7>;
            case 8: return (const void*)bwd_tile_kernel<T, 8>;
            default: return nullptr;
        }
    }
}

// Block path: cols <= 16384 and 512 threads give at most 4 vectors per thread for bf16 and
// 8 for fp32.  Kahan compensation when a thread owns at most 16 columns.
template <typename T>
const void* block_kernel(int vpt) {
    if constexpr (Io<T>::kVec == 8) {
        switch (vpt) {
            case 1: return (const void*)bwd_block_kernel<T, 1, true>;
            case 2: return (const void*)bwd_block_kernel<T, 2, true>;
            case 3: return (const void*)bwd_block_kernel<T, 3, false>;
            case 4: return (const void*)bwd_block_kernel<T, 4, false>;
            default: return nullptr;
        }
    } else {
        switch (vpt) {
            case 1: return (const void*)bwd_block_kernel<T, 1, true>;
            case 2: return (const void*)bwd_block_kernel<T, 2, true>;
            case 3: return (const void*)bwd_block_kernel<T, 3, true>;
            case 4: return (const void*)bwd_block_kernel<T, 4, true>;
            case 5: return (const void*)bwd_block_kernel<T, 5, false>;
            case 6: return (const void*)bwd_block_kernel<T, 6, false>;
            case 7: return (const void*)bwd_block_kernel<T, 7, false>;
            case 8: return (const void*)bwd_block_kernel<T, 8, false>;
            default: return nullptr;
        }
    }
}

const void* kernel_for(Dtype dt, const BwdPlan& p) {
    const bool f = dt == Dtype::F32;
    if (p.path == kPathWarp) return f ? warp_kernel<float>(p.per_thread) : warp_kernel<__nv_bfloat16>(p.per_thread);
    if (p.path == kPathBlock) return f ? block_kernel<float>(p.per_thread) : block_kernel<__nv_bfloat16>(p.per_thread);
    return f ? (const void*)bwd_scalar_kernel<float> : (const void*)bwd_scalar_kernel<__nv_bfloat16>;
}

// Number of finishing blocks: enough that each finishing thread adds about 8 partial
// vectors, and no more than there are blocks or column groups.
int pick_finishers(int grid, int cols, int threads) {
    const int U = cols % 2 == 0 ? 2 : 1;
    const int ngroups = cols / U;
    const int want_q = std::max(1, (grid + 7) / 8);
    const int units_max = std::max(2, threads / want_q);
    const int wg_max = std::max(1, units_max / 2);
    int F = (ngroups + wg_max - 1) / wg_max;
    F = std::max(1, std::min(F, std::min(grid, ngroups)));
    return F;
}

}  // namespace

int bwd_max_grid(int rows, int sms) { return std::max(1, std::min(rows, sms * 8)); }

cudaError_t plan_bwd(Dtype dt, int rows, int cols, bool aligned, int path_override,
                     BwdPlan* plan) {
    const DeviceInfo& di = device_info(-1);
    const int V = dt == Dtype::F32 ? 4 : 8;
    const int esize = dt == Dtype::F32 ? 4 : 2;
    BwdPlan p;
    if (aligned && path_override != kPathScalar) {
        const int nvec = cols / V;
        const int vpl = (nvec + 31) / 32;
        const int warp_max = dt == Dtype::F32 ? 8 : 5;
        const bool warp_fits = vpl <= warp_max;
        const bool warp_auto = dt == Dtype::BF16 && rows <= kWarpPathMaxRows;
        if (warp_fits && (path_override == kPathWarp ||
                          (path_override == kPathAuto && warp_auto))) {
            p.path = kPathWarp;
            p.per_thread = vpl;
            p.threads = kTileThreads;
            const size_t slot = 2ull * kTileRows * cols * esize;  // a tile of dy and of x
            int stages = (int)std::min<size_t>(kMaxStages, ((size_t)di.smem_optin / 2) / slot);
            stages = std::max(2, stages);
            p.stages = stages;
            // The ring, reused afterwards for the warps' sums and the finish scratch.
            p.smem = std::max<size_t>({(size_t)stages * slot, (size_t)kTileRows * cols * 4,
                                       (size_t)kTileThreads * 16});
        } else {
            p.path = kPathBlock;
            p.per_thread = (nvec + kBwdBlockMaxThreads - 1) / kBwdBlockMaxThreads;
            const int t = (nvec + p.per_thread - 1) / p.per_thread;
            p.threads = std::max(32, (t + 31) / 32 * 32);
            const size_t slot = 2ull * cols * esize;
            const size_t budget = std::max<size_t>(slot, (size_t)di.smem_optin / 2);
            int stages = (int)std::min<size_t>(kMaxStages, budget / slot);
            stages = std::max(1, stages);
            p.smem = std::max<size_t>((size_t)stages * slot, (size_t)p.threads * 16);
            p.stages = stages;
        }
    } else {
        p.path = kPathScalar;
        p.threads = kBwdScalarThreads;
        const size_t acc = 16ull * cols;  // (hi, lo) pairs for both statistics
        const bool fits = acc <= (size_t)di.smem_optin / 2;
        p.smem = std::max<size_t>(fits ? acc : 0, (size_t)kBwdScalarThreads * 16);
        p.stages = fits ? 1 : 0;  // tells the kernel where its accumulators live
    }
    if (p.smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
    const void* kern = kernel_for(dt, p);
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    const int occ = blocks_per_sm(kern, p.threads, p.smem);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int need = p.path == kPathWarp ? (rows + kTileRows - 1) / kTileRows : rows;
    p.grid = std::max(1, std::min(need, di.sms * occ));
    p.finishers = pick_finishers(p.grid, cols, p.threads);
    *plan = p;
    return cudaSuccess;
}

cudaError_t launch_bwd(Dtype dt, const BwdArgs& a, const BwdPlan& p, cudaStream_t stream,
                       int* launches) {
    *launches = 0;
    const void* kern = kernel_for(dt, p);
    if (!kern) return cudaErrorInvalidValue;
    KParams k;
    k.dy = a.dy;
    k.xr = a.xr;
    k.gamma = a.gamma;
    k.mean = a.mean;
    k.rstd = a.rstd;
    k.dx = a.dx;
    k.dgamma = a.dgamma;
    k.dbeta = a.dbeta;
    k.rows = a.rows;
    k.cols = a.cols;
    k.part = reinterpret_cast<float2*>(a.partials);
    k.ctr = a.counters;
    k.status = a.status;
    k.limit_ns = a.wait_limit_ns;
    k.wait_extra = a.wait_extra;
    k.finishers = p.finishers;
    k.stages = p.stages;
    void* args[] = {&k};
    // A cooperative launch (all blocks co-resident, checked by the driver against the
    // occupancy), issued through cudaLaunchKernelEx so that it can also be captured into a
    // CUDA graph.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
