// ln_bwd_kernels.cuh -- backward kernels of the fused residual-add + LayerNorm (and, with
// RMS = true, of the fused residual-add + RMSNorm), and their launch planning.  Included by
// ln_bwd.cu (LayerNorm instantiations) and rms_bwd.cu (RMSNorm instantiations), so that the
// two sets compile in parallel.
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
//  1. Each block owns a FIXED set of rows (every G-th row or tile of rows; a contiguous range
//     in the scalar kernel).  While it computes dx it
//     accumulates dy * xhat and dy for the columns its threads own and, at the end, writes
//     one row of partial sums per statistic to the workspace: part[stat][block][col].
//  2. The blocks that own a slice of the columns then read every block's partials of their
//     slice, add them over blocks in a fixed order and write dgamma and dbeta; the others
//     leave.  A partial announces itself: the workspace words are zero between calls and a
//     stored partial never is (see part_enc), so a reader polls, bounded, only the words it
//     is still missing -- no fence, arrival counter or grid-wide wait -- and zeroes what it
//     has read for the next call.
//  This is the last-block-finishes idea of llm.c's layernorm_backward_kernel10 ("llm.c: the
//  llmc/ CUDA kernel layer", section 3.3), widened from one finishing block to many so that
//  the finish is spread over SMs instead of serialising one SM on all partials.  The warp
//  and scalar kernels finish in the same launch, which is cooperative, so every block is
//  resident and the polls always end; the block-per-row kernel hands the finish to a second
//  launch that waits for it to complete (programmatic dependent launch), so nothing polls
//  there.  Which block adds which rows, and in what order, depends only on (rows, cols,
//  device), so dgamma and dbeta are bitwise reproducible run to run.
//
// Accuracy of the column sums.  A plain fp32 sum of n terms of size sigma carries an error
// of about 2^-24 * sigma * sqrt(n * L) for chains of L additions, whatever the order: for
// 262144 rows that is ~1e-4, far above the 2e-5 that fp32 results are held to.  So for fp32
// I/O (and bf16 rows long enough to make chains long) each thread or lane keeps its running
// sums compensated (Kahan: a second fp32 register holds the rounding error of every
// addition), partial sums are stored as (hi, lo) fp32 pairs and every later addition is
// error-free (TwoSum), so the only rounding left is the final one to the output type.  For
// bf16 results over short chains plain fp32 sums are far more accurate than the bf16 unit
// in the last place, and the partials are stored and added plainly.
#pragma once

#include <algorithm>
#include <climits>
#include <type_traits>

#include "ln_device.cuh"
#include "ln_finish.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

// Consumer warps = rows per tile, plus one producer warp: 8 warps, because registers are
// allocated to warps in groups of four (a 9-warp block would pay for 12).
constexpr int kTileRows = 7;
constexpr int kTileThreads = (kTileRows + 1) * 32;

// Rows per tile of the tile kernel with W warps per row (rows wider than one warp's share
// of registers).  One block per SM; its consumer warps + the producer are as many as the
// registers allow: a thread keeps gamma and the column sums of VPL vectors (H fp32 pairs
// each; the sums compensated when KAHAN) plus ~56 registers of working state, and warps
// are paid for in fours.
__host__ __device__ constexpr int tile_rows_for(int H, int vpl, bool kahan, int W) {
    if (W == 1) return kTileRows;
    const int regs = 2 * (kahan ? 5 : 3) * vpl * H + 56;
    const int warps = (65536 / (32 * ((regs + 7) / 8 * 8))) / 4 * 4;
    return (warps - 1) / W > 1 ? (warps - 1) / W : 1;
}
template <typename T, int VPL, bool KAHAN, int W>
constexpr int tile_threads() {
    return (tile_rows_for(Pairs<T>::kPairs, VPL, KAHAN, W) * W + 1) * 32;
}
constexpr int kBwdBlockMaxThreads = 512;
constexpr int kBwdScalarThreads = 256;
constexpr int kMaxStages = 8;
constexpr int kBlockStages = 3;
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
    float2* part;  // [2][gridDim.x][cols] (hi, lo) pairs, or plain fp32 sums when compact
    float2* acc;   // scalar kernel, rows too wide for shared memory: its running (hi, lo) sums
    int compact;   // partials without the lo half (kernels whose column sums are plain)
    int fin_rw;    // warps per unit group in the finish (divides the block's warp count)
    int nstat;     // column statistics: 2 (dgamma, dbeta) or 1 (the RMSNorm's dgamma)
    int P;         // partial rows (the row kernel's grid)
    int split_finish;  // 1: a separate dependent launch finishes; 0: the row kernel does
    unsigned* ctr;  // a zero word nothing writes (the bounded-wait test polls it)
    unsigned* status;
    uint64_t limit_ns;
    unsigned wait_extra;
    int stages;
};

// This block's share [r0, r1) of n items split over the grid: the first n % G blocks take
// one item more (32-bit arithmetic: one division, no 64-bit products).
__device__ __forceinline__ void row_range(int n, int& r0, int& r1) {
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int q = n / G, rem = n - q * G;
    r0 = b * q + min(b, rem);
    r1 = r0 + q + (b < rem ? 1 : 0);
}

// Kahan step on fp32 pairs: the running value is s - c.
__device__ __forceinline__ void kahan2(f2& s, f2& c, f2 x) {
    const f2 y = f2_sub(x, c);
    const f2 t = f2_add(s, y);
    c = f2_sub(f2_sub(t, s), y);
    s = t;
}

// Kahan step: the running value is s - c.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

// The finish of block f of F over P partial rows, for the partial layout the plan chose.
template <typename T>
__device__ void finish_dispatch(const KParams& a, int P, int F, int f, float* scratch) {
    if (a.compact) {
        if (a.cols % 4 == 0)
            finish_units<T, 4, true>(a, P, F, f, scratch);
        else if (a.cols % 2 == 0)
            finish_units<T, 2, true>(a, P, F, f, scratch);
        else
            finish_units<T, 1, true>(a, P, F, f, scratch);
    } else {
        if (a.cols % 2 == 0)
            finish_units<T, 2, false>(a, P, F, f, scratch);
        else
            finish_units<T, 1, false>(a, P, F, f, scratch);
    }
}

// Unit groups of the finish (as finish_units splits them).
__device__ __forceinline__ int finish_groups(const KParams& a) {
    const int U = a.compact ? (a.cols % 4 == 0 ? 4 : a.cols % 2 == 0 ? 2 : 1)
                            : (a.cols % 2 == 0 ? 2 : 1);  // as finish_dispatch instantiates
    return (a.nstat * (a.cols / U) + kFinUnits - 1) / kFinUnits;
}

// Called by every thread of every block once the block's partial row is stored, when the
// finish runs inside the row kernel.  Blocks that own no unit group of the finish are done
// and leave, freeing their SM; the others finish their groups, picking up each block's
// partials as they land.
template <typename T>
__device__ void finish_if_owner(const KParams& a, float* scratch) {
    if (a.split_finish) return;  // a separate launch finishes
    const int P = (int)gridDim.x, f = (int)blockIdx.x;
    const int ng = finish_groups(a);
    const bool finisher = (f + 1) * ng / P > f * ng / P;  // as finish_units splits the groups
    if (!finisher) return;  // the same for every thread of the block
    __syncthreads();        // shared memory becomes the finish's scratch
    if (a.wait_extra && threadIdx.x == 0) {
        // Test hook: also wait for a word that nothing writes, so the limit runs out.
        if (!wait_counter_geq(a.ctr, 1u, a.limit_ns)) raise_status(a.status, kStatusTimeout);
    }
    finish_dispatch<T>(a, P, P, f, scratch);
}

// The finish as its own launch, programmatically dependent on the row kernel: its blocks are
// scheduled while the row kernel runs and wait (griddepcontrol.wait) until it has completed,
// so every partial row is already written when they read them -- no polling.
constexpr int kFinThreads = 256;
template <typename T>
__global__ void __launch_bounds__(kFinThreads) bwd_finish_kernel(const KParams a) {
    __shared__ float scratch[kFinThreads * 8];  // 2 U floats per thread, U <= 4
    pdl_enter();
    if (a.wait_extra && threadIdx.x == 0) {
        if (!wait_counter_geq(a.ctr, 1u, a.limit_ns)) raise_status(a.status, kStatusTimeout);
    }
    finish_dispatch<T>(a, a.P, (int)gridDim.x, (int)blockIdx.x, scratch);
}

// ---------------------------------------------------------------------------------------
// Warp per row, fed by a bulk-copy (TMA) pipeline (the forward's tile kernel, for dy and x).
// The block owns a fixed set of tiles (RT consecutive rows each, every G-th); the producer
// warp's lane 0 fetches each tile of dy and of x with one cp.async.bulk apiece, `stages`
// tiles ahead; consumer warp w handles row w of every tile.  Lane l owns the columns of
// vectors l, l+32, ... in every row, so its column sums stay in registers (Kahan-compensated
// when KAHAN, for fp32 I/O and for long chains of rows); at the end the consumer warps'
// sums are added in warp order with TwoSum through shared memory (the drained ring) into
// the block's (hi, lo) partial row.
// Rows too wide for one warp's registers (W = 2 or 4): W warps share each row of the tile,
// lane l of warp p taking vectors (v * W + p) * 32 + l, and add their two row sums in warp
// order after exchanging them through shared memory (each warp announces its pair on an
// mbarrier; bounded waits).  The block then keeps RT rows in flight at once instead of one
// (the block-per-row kernel): bf16 8192 x 2560 backward 44.0 -> 31.7 us, 8192 x 2048
// 28.0 -> 23.4 us, fp32 8192 x 1280 41.3 -> 28.9 us, measured on GB300.
// ---------------------------------------------------------------------------------------
// Two blocks per SM when the per-lane state (gamma, column sums and their compensations,
// in fp32 pairs) leaves room: at most 128 registers per thread.
template <typename T, int VPL, bool KAHAN>
constexpr int tile_min_blocks() {
    return (KAHAN ? 5 : 3) * VPL * Pairs<T>::kPairs <= 36 ? 2 : 1;
}

template <typename T, int VPL, bool KAHAN, bool RMS, int W = 1>
__global__ void __launch_bounds__(tile_threads<T, VPL, KAHAN, W>(),
                                  W == 1 ? tile_min_blocks<T, VPL, KAHAN>() : 1)
    bwd_tile_kernel(const KParams a) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    // RT rows per tile, W warps per row: consumer warp c takes row c / W of every tile and,
    // in it, the vectors (v * W + c % W) * 32 + lane.
    constexpr int RT = tile_rows_for(Pairs<T>::kPairs, VPL, KAHAN, W);
    constexpr int NCW = RT * W;  // consumer warps; warp NCW is the producer
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    // W > 1: the W warps of a row exchange their two row sums through xval, announced on
    // xbar (one barrier per row of the tile, double-buffered by step parity).
    __shared__ uint64_t xbar[W > 1 ? 2 * RT : 1];
    __shared__ float2 xval[W > 1 ? 2 * RT * W : 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wrow = warp / W, wpos = warp - wrow * W;  // row of the tile, place in the row
    const int lane_vec = wpos * 32 + lane;              // this lane's first vector of a row
    constexpr int VSTRIDE = 32 * W;                     // between a lane's vectors
    const int cols = a.cols, nvec = cols / V, stages = a.stages, rows = a.rows;
    const RowDivisor rdiv(cols);
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned tile_bytes = (unsigned)RT * row_bytes;
    const unsigned slot_bytes = 2u * tile_bytes;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    // This block's tiles: b, b + G, b + 2G, ... (G blocks).  Interleaved rather than a
    // contiguous range, so the first tiles every block requests are the first tiles of the
    // tensor and the DRAM queue serves all blocks evenly (measured on GB300: bf16 8192x1280
    // backward 18.4 -> 17.8 us).  The assignment depends only on (rows, cols, device).
    const int ntiles = (rows + RT - 1) / RT;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int my_tiles = b < ntiles ? (ntiles - 1 - b) / G + 1 : 0;
    auto tile_row0 = [&](int k) { return (b + k * G) * RT; };  // first row of step k

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], NCW);
        }
        if constexpr (W > 1)
            for (int i = 0; i < 2 * RT; ++i) mbar_init(&xbar[i], W);
        fence_barrier_init();
    }
    __syncthreads();
    // Set-up done; nothing above touches global memory, so it overlaps the previous grid.
    pdl_enter();

    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    constexpr int KV = KAHAN ? VPL : 1;
    f2 accg[VPL][H], accb[VPL][H];  // this lane's column sums of dy * xhat and dy
    f2 cmpg[KV][H], cmpb[KV][H];    // their Kahan compensations (the value is s - c)
#pragma unroll
    for (int v = 0; v < VPL; ++v)
#pragma unroll
        for (int h = 0; h < H; ++h) accg[v][h] = accb[v][h] = f2_splat(0.f);
#pragma unroll
    for (int v = 0; v < KV; ++v)
#pragma unroll
        for (int h = 0; h < H; ++h) cmpg[v][h] = cmpb[v][h] = f2_splat(0.f);

    if (warp == NCW) {  // producer
        if (lane == 0) {
            int k = 0;
            RingPos pos;
            for (; k < my_tiles; ++k, pos.next(stages)) {
                const int slot = pos.slot;
                // With a 2-slot ring (two blocks per SM) the second tile is requested once the
                // first has landed, so every block's first tile is ahead of all second tiles
                // in the DRAM queue and the late blocks start sooner (measured on GB300: bf16
                // 8192x768 backward 12.6 -> 12.2 us; with a 4-slot ring, one block per SM,
                // holding back the rest of the first fill was slower: bf16 8192x1280
                // 16.3 -> 17.2 us).  A timeout here shows again in the consumers' wait.
                if (k == 1 && stages == 2) (void)mbar_wait(&full_bar[0], 0u, a.limit_ns);
                // A slot's second and later fills wait for the consumers of the previous pass.
                if (k >= stages && !mbar_wait(&empty_bar[slot], pos.phase ^ 1u, a.limit_ns)) {
                    raise_status(a.status, kStatusTimeout);
                    break;
                }
                const int r0 = tile_row0(k);
                const unsigned bytes = (unsigned)min(RT, rows - r0) * row_bytes;
                unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
                mbar_arrive_expect_tx(&full_bar[slot], 2u * bytes);
                bulk_g2s(dst, dy + (size_t)r0 * cols, bytes, &full_bar[slot]);
                bulk_g2s(dst + tile_bytes, xr + (size_t)r0 * cols, bytes, &full_bar[slot]);
            }
            for (int j = max(0, k - stages); j < k; ++j)  // drain: every copy has landed
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, a.limit_ns);
        }
    } else {  // consumers
        f2 gm[VPL][H];  // gamma of this lane's columns as fp32 pairs, loaded once
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const int vi = v * VSTRIDE + lane_vec;
            PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gm[v]);
        }
        int xstep = 0;    // W > 1: rows this warp has exchanged sums for (buffer and phase)
        bool xok = true;  // W > 1: the row's other warps announced their sums in time
        // One or two rows through both passes.  With two (the warp's row of tile k and of
        // tile k + 1), their first passes run together, their four row sums share one
        // butterfly and their second passes run together; per lane the column sums still add
        // tile k's terms before tile k + 1's, so the results are those of one row at a time.
        auto body = [&](auto nr_c, const int (&row_)[2], const int (&slot_)[2],
                        const float (&mu_)[2], const float (&rs_)[2]) {
            constexpr int NR = decltype(nr_c)::value;
            const T* dys[NR];
            const T* xs[NR];
            f2 mu2[NR], rs2[NR], sg[NR], sgx[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                dys[r] = reinterpret_cast<const T*>(smem_raw + (size_t)slot_[r] * slot_bytes +
                                                    (size_t)wrow * row_bytes);
                xs[r] = dys[r] + (size_t)RT * cols;
                mu2[r] = f2_splat(mu_[r]);
                rs2[r] = f2_splat(rs_[r]);
                // Row sums; the low halves take the even columns, the high halves the odd.
                sg[r] = sgx[r] = f2_splat(0.f);
            }
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * VSTRIDE + lane_vec;
                if (vi < nvec) {
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        f2 d[H], xx[H];
                        PR::load_staged(dys[r] + (size_t)vi * V, d);
                        PR::load_staged(xs[r] + (size_t)vi * V, xx);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const f2 xh = f2_mul(f2_sub(xx[h], mu2[r]), rs2[r]);
                            const f2 g = f2_mul(gm[v][h], d[h]);
                            if constexpr (!RMS) sg[r] = f2_add(sg[r], g);
                            sgx[r] = f2_fma(g, xh, sgx[r]);
                            if constexpr (KAHAN) {
                                kahan2(accg[v][h], cmpg[v][h], f2_mul(d[h], xh));
                                if constexpr (!RMS) kahan2(accb[v][h], cmpb[v][h], d[h]);
                            } else {
                                accg[v][h] = f2_fma(d[h], xh, accg[v][h]);
                                if constexpr (!RMS) accb[v][h] = f2_add(accb[v][h], d[h]);
                            }
                        }
                    }
                }
            }
            // The one reduction of each row: both of its sums together (xor butterfly).  The
            // RMSNorm has one sum per row (its mean term is zero): two rows share a butterfly.
            float t[2 * NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                t[2 * r] = RMS ? 0.f : f2_lo(sg[r]) + f2_hi(sg[r]);
                t[2 * r + 1] = f2_lo(sgx[r]) + f2_hi(sgx[r]);
            }
            if constexpr (RMS) {
                if constexpr (NR == 2)
                    warp_sum2(t[1], t[3]);
                else
                    warp_sum2(t[1], t[0]);
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) warp_sum2(t[2 * r], t[2 * r + 1]);
            }
            if constexpr (W > 1) {  // one row (NR = 1): add the W warps' sums in warp order
                const int xi = (xstep & 1) * RT + wrow;
                if (lane == 0) {
                    xval[xi * W + wpos] = make_float2(t[0], t[1]);
                    mbar_arrive(&xbar[xi]);
                }
                xok = __all_sync(kFullMask, mbar_wait(&xbar[xi], (unsigned)(xstep >> 1) & 1u, a.limit_ns));
                ++xstep;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int j = 0; j < W; ++j) {
                    const float2 q = xval[xi * W + j];
                    s0 += q.x;
                    s1 += q.y;
                }
                t[0] = s0;
                t[1] = s1;
            }
            // dx = rs * (g - (mg + xhat * mgx)) with the same rounded g as in the sums, so
            // g - mg cancels exactly where it should (a one-column row gives dx = 0); mg = 0
            // for the RMSNorm.
            f2 mg2[NR], mgx2[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                mg2[r] = f2_splat(RMS ? 0.f : rdiv.div(t[2 * r]));
                mgx2[r] = f2_splat(rdiv.div(t[2 * r + 1]));
            }
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * VSTRIDE + lane_vec;
                if (vi < nvec) {  // second pass re-reads the rows from shared memory
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        f2 d[H], xx[H], o[H];
                        PR::load_staged(dys[r] + (size_t)vi * V, d);
                        PR::load_staged(xs[r] + (size_t)vi * V, xx);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const f2 xh = f2_mul(f2_sub(xx[h], mu2[r]), rs2[r]);
                            const f2 g = f2_mul(gm[v][h], d[h]);
                            o[h] = f2_mul(rs2[r], f2_sub(g, f2_fma(xh, mgx2[r], mg2[r])));
                        }
                        st_stream(dx + (size_t)row_[r] * cols + (size_t)vi * V, PR::pack(o));
                    }
                }
            }
        };
        // Rows go in pairs of consecutive tiles when the ring is deep enough that the pair's
        // two slots still leave tiles in flight behind them.  The paired form is built for
        // bf16 rows of 4 or 5 vectors per lane and for fp32 rows, where it measured faster on
        // GB300 (bf16 8192x1280: 21.8 -> 19.9 us; fp32 262144x1000: 544 -> 507 us, there
        // even at ring depths that keep it to one row at a time); bf16 rows of 3 or fewer
        // vectors per lane measured slower with it.
        constexpr bool kPairRows = W == 1 && ((Io<T>::kVec == 8 && VPL >= 4) || Io<T>::kVec == 4);
        const int pair_max = (kPairRows && stages >= 4) ? 2 : 1;
        // mean and rstd of the next step's rows are loaded a step ahead, so their latency is
        // not on the rows' critical path.
        auto load_stats = [&](int kk, int nr, float (&mu)[2], float (&rs)[2]) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rr = tile_row0(kk + r) + wrow;
                const bool valid = r < nr && kk + r < my_tiles && rr < rows;
                mu[r] = valid && !RMS ? a.mean[rr] : 0.f;  // the RMSNorm subtracts no mean
                rs[r] = valid ? a.rstd[rr] : 0.f;
            }
        };
        float mu_n[2], rs_n[2];
        load_stats(0, min(pair_max, my_tiles), mu_n, rs_n);
        RingPos pos;
        for (int k = 0; k < my_tiles;) {
            const int nr = min(pair_max, my_tiles - k);
            int slots[2];
            unsigned phases[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                slots[r] = pos.slot;
                phases[r] = pos.phase;
                if (r < nr) pos.next(stages);
            }
            const float mu[2] = {mu_n[0], mu_n[1]}, rs[2] = {rs_n[0], rs_n[1]};
            if (k + nr < my_tiles) load_stats(k + nr, min(pair_max, my_tiles - k - nr), mu_n, rs_n);
            bool ok = mbar_wait(&full_bar[slots[0]], phases[0], a.limit_ns);
            if (nr == 2) ok = mbar_wait(&full_bar[slots[1]], phases[1], a.limit_ns) && ok;
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) raise_status(a.status, kStatusTimeout);
                break;
            }
            const int rws[2] = {tile_row0(k) + wrow, tile_row0(k + 1) + wrow};
            if constexpr (kPairRows) {
                if (nr == 2 && rws[1] < rows)
                    body(std::integral_constant<int, 2>{}, rws, slots, mu, rs);
                else if (rws[0] < rows)
                    body(std::integral_constant<int, 1>{}, rws, slots, mu, rs);
            } else if (rws[0] < rows) {
                body(std::integral_constant<int, 1>{}, rws, slots, mu, rs);
            }
            if (!xok) {  // (W > 1) a warp of this row stopped: stop too, bounded
                if (lane == 0) raise_status(a.status, kStatusTimeout);
                break;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty_bar[slots[0]]);
                if (nr == 2) mbar_arrive(&empty_bar[slots[1]]);
            }
            k += nr;
        }
    }
    __syncthreads();  // the ring is drained and no warp reads it any more

    // Block partial row.  The consumer warps put their sums in shared memory as
    // [stat][row of the tile][cols] floats (the drained ring; the W warps of a row own
    // disjoint columns), followed by the negated compensations in the same layout when
    // KAHAN; then each thread adds the RT rows' values of a group of 4 columns in order (with
    // TwoSum when KAHAN) and stores the block's partials of them.
    float* smem_f = reinterpret_cast<float*>(smem_raw);
    const size_t lo_off = (size_t)2 * RT * cols;
    auto put = [&](float* dst, f2 a0, f2 a1) {
        *reinterpret_cast<float4*>(dst) = make_float4(f2_lo(a0), f2_hi(a0), f2_lo(a1), f2_hi(a1));
    };
    if (warp < NCW) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const int vi = v * VSTRIDE + lane_vec;
            if (vi < nvec) {
                float* dg = smem_f + (size_t)wrow * cols + (size_t)vi * V;
                float* db = dg + (size_t)RT * cols;
                const f2 z = f2_splat(0.f);
                if constexpr (H == 4) {
                    // A lane's 8 columns are two 16-byte halves at a 32-byte lane stride.
                    // Lanes 4-7 of each group of 8 store their upper half first, so the 8
                    // lanes of a 128-bit store phase hit 8 distinct groups of 4 banks.
                    const bool sw = ((lane >> 2) & 1) != 0;
                    const int o0 = sw ? 4 : 0, o1 = sw ? 0 : 4;
                    put(dg + o0, sw ? accg[v][2] : accg[v][0], sw ? accg[v][3] : accg[v][1]);
                    put(dg + o1, sw ? accg[v][0] : accg[v][2], sw ? accg[v][1] : accg[v][3]);
                    if constexpr (!RMS) {
                        put(db + o0, sw ? accb[v][2] : accb[v][0], sw ? accb[v][3] : accb[v][1]);
                        put(db + o1, sw ? accb[v][0] : accb[v][2], sw ? accb[v][1] : accb[v][3]);
                    }
                    if constexpr (KAHAN) {
                        put(dg + lo_off + o0, f2_sub(z, sw ? cmpg[v][2] : cmpg[v][0]),
                            f2_sub(z, sw ? cmpg[v][3] : cmpg[v][1]));
                        put(dg + lo_off + o1, f2_sub(z, sw ? cmpg[v][0] : cmpg[v][2]),
                            f2_sub(z, sw ? cmpg[v][1] : cmpg[v][3]));
                        if constexpr (!RMS) {
                            put(db + lo_off + o0, f2_sub(z, sw ? cmpb[v][2] : cmpb[v][0]),
                                f2_sub(z, sw ? cmpb[v][3] : cmpb[v][1]));
                            put(db + lo_off + o1, f2_sub(z, sw ? cmpb[v][0] : cmpb[v][2]),
                                f2_sub(z, sw ? cmpb[v][1] : cmpb[v][3]));
                        }
                    }
                } else {  // fp32: one 16-byte store per vector, consecutive lanes adjacent
                    put(dg, accg[v][0], accg[v][1]);
                    if constexpr (!RMS) put(db, accb[v][0], accb[v][1]);
                    if constexpr (KAHAN) {
                        put(dg + lo_off, f2_sub(z, cmpg[v][0]), f2_sub(z, cmpg[v][1]));
                        if constexpr (!RMS) put(db + lo_off, f2_sub(z, cmpb[v][0]), f2_sub(z, cmpb[v][1]));
                    }
                }
            }
        }
    }
    __syncthreads();
    const int P = gridDim.x;
    const int quarter = cols >> 2;  // groups of 4 columns per statistic (cols is a multiple of 4)
    for (int u = tid; u < (RMS ? 1 : 2) * quarter; u += blockDim.x) {
        const int stat = u >= quarter ? 1 : 0;
        const int c = 4 * (u - stat * quarter);
        const float* src = smem_f + (size_t)stat * RT * cols + c;
        if constexpr (KAHAN) {
            float S[4] = {0.f, 0.f, 0.f, 0.f}, C[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < RT; ++w) {
                const float4 t = *reinterpret_cast<const float4*>(src + (size_t)w * cols);
                const float4 l = *reinterpret_cast<const float4*>(src + lo_off + (size_t)w * cols);
                comp_add(S[0], C[0], t.x, l.x);
                comp_add(S[1], C[1], t.y, l.y);
                comp_add(S[2], C[2], t.z, l.z);
                comp_add(S[3], C[3], t.w, l.w);
            }
            float4* dst = reinterpret_cast<float4*>(a.part + ((size_t)stat * P + blockIdx.x) * cols + c);
            st_part4(dst, S[0], C[0], S[1], C[1]);
            st_part4(dst + 1, S[2], C[2], S[3], C[3]);
        } else {  // plain fp32 sums feeding a bf16 result: a few more additions are noise
            f2 S01 = f2_splat(0.f), S23 = f2_splat(0.f);
#pragma unroll
            for (int w = 0; w < RT; ++w) {
                const float4 t = *reinterpret_cast<const float4*>(src + (size_t)w * cols);
                S01 = f2_add(S01, f2_make(t.x, t.y));
                S23 = f2_add(S23, f2_make(t.z, t.w));
            }
            st_part4(reinterpret_cast<float*>(a.part) + ((size_t)stat * P + blockIdx.x) * cols + c,
                     f2_lo(S01), f2_hi(S01), f2_lo(S23), f2_hi(S23));
        }
    }
    finish_if_owner<T>(a, smem_f);
}

// ---------------------------------------------------------------------------------------
// Block per row with bulk-copy staging of dy and x rows (several rows ahead).  Thread t of
// the block (blockDim.x threads) owns the columns of vectors t, t + blockDim.x, ... in
// every row, so its column sums stay in registers (compensated when KAHAN) and go straight
// to the block's partial row.
// ---------------------------------------------------------------------------------------
template <typename T, int VPT, bool KAHAN, bool RMS>
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
    const RowDivisor rdiv(cols);
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned slot_bytes = 2u * row_bytes;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    // This block's rows: b, b + G, b + 2G, ... (G blocks), interleaved as in the tile kernel.
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int nmy = b < a.rows ? (a.rows - 1 - b) / G + 1 : 0;

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&full_bar[i], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Set-up done; nothing above touches global memory, so it overlaps the previous grid.
    pdl_enter();
    auto issue = [&](int k, int slot) {  // thread 0 only: fetch the block's k-th row into `slot`
        if (k >= nmy) return;
        const int row = b + k * G;
        unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], slot_bytes);
        bulk_g2s(dst, dy + (size_t)row * cols, row_bytes, &full_bar[slot]);
        bulk_g2s(dst + row_bytes, xr + (size_t)row * cols, row_bytes, &full_bar[slot]);
    };
    if (tid == 0)
        for (int k = 0; k < stages; ++k) issue(k, k);

    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    constexpr int KV = KAHAN ? VPT : 1;
    f2 gp[VPT][H];            // gamma of this thread's columns as fp32 pairs
    f2 sg[VPT][H], sb[VPT][H];  // running column sums of dy * xhat and dy
    f2 cg[KV][H], cb[KV][H];    // their Kahan compensations (the value is s - c)
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = v * nthreads + tid;
        PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gp[v]);
#pragma unroll
        for (int h = 0; h < H; ++h) sg[v][h] = sb[v][h] = f2_splat(0.f);
    }
#pragma unroll
    for (int v = 0; v < KV; ++v)
#pragma unroll
        for (int h = 0; h < H; ++h) cg[v][h] = cb[v][h] = f2_splat(0.f);

    int k = 0;
    // mean and rstd are loaded one row ahead (off the row's critical path).
    // (The RMSNorm subtracts no mean: mu = 0 makes xhat = x * rs exactly.)
    float mu_next = nmy > 0 && !RMS ? a.mean[b] : 0.f, rs_next = nmy > 0 ? a.rstd[b] : 0.f;
    RingPos pos;
    for (int row = b; k < nmy; row += G, ++k, pos.next(stages)) {
        const int slot = pos.slot;
        const float mu = mu_next, rs = rs_next;
        if (k + 1 < nmy) {
            if constexpr (!RMS) mu_next = a.mean[row + G];
            rs_next = a.rstd[row + G];
        }
        if (!mbar_wait(&full_bar[slot], pos.phase, a.limit_ns)) abort_flag = 1;
        const T* dys = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes);
        const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes + row_bytes);
        const size_t base = (size_t)row * cols;
        const f2 mu2 = f2_splat(mu), rs2 = f2_splat(rs);
        f2 rg = f2_splat(0.f), rgx = f2_splat(0.f);  // row sums: even columns low, odd high
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                f2 d[H], xx[H];
                PR::load_staged(dys + (size_t)vi * V, d);
                PR::load_staged(xs + (size_t)vi * V, xx);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const f2 xh = f2_mul(f2_sub(xx[h], mu2), rs2);
                    const f2 g = f2_mul(gp[v][h], d[h]);
                    if constexpr (!RMS) rg = f2_add(rg, g);
                    rgx = f2_fma(g, xh, rgx);
                    if constexpr (KAHAN) {
                        kahan2(sg[v][h], cg[v][h], f2_mul(d[h], xh));
                        if constexpr (!RMS) kahan2(sb[v][h], cb[v][h], d[h]);
                    } else {
                        sg[v][h] = f2_fma(d[h], xh, sg[v][h]);
                        if constexpr (!RMS) sb[v][h] = f2_add(sb[v][h], d[h]);
                    }
                }
            }
        }
        float tg = f2_lo(rg) + f2_hi(rg), tgx = f2_lo(rgx) + f2_hi(rgx);
        warp_sum2(tg, tgx);
        if (lane == 0) {
            red[0][warp] = tg;
            red[1][warp] = tgx;
        }
        __syncthreads();  // the one cross-warp exchange of the row
        if (abort_flag) break;
        sum_warp_values2(red[0], red[1], nw, tg, tgx);  // the same bits in every thread
        const f2 mg2 = f2_splat(RMS ? 0.f : rdiv.div(tg)), mgx2 = f2_splat(rdiv.div(tgx));
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                f2 d[H], xx[H], o[H];
                PR::load_staged(dys + (size_t)vi * V, d);
                PR::load_staged(xs + (size_t)vi * V, xx);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const f2 xh = f2_mul(f2_sub(xx[h], mu2), rs2);
                    const f2 g = f2_mul(gp[v][h], d[h]);
                    o[h] = f2_mul(rs2, f2_sub(g, f2_fma(xh, mgx2, mg2)));
                }
                st_stream(dx + base + (size_t)vi * V, PR::pack(o));
            }
        }
        __syncthreads();  // slot and `red` free again
        if (tid == 0) issue(k + stages, slot);  // row k + stages takes row k's slot
    }

    if (abort_flag) {
        if (tid == 0) {
            raise_status(a.status, kStatusTimeout);
            for (int j = k; j < k + stages && j < nmy; ++j)
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, a.limit_ns);
        }
        __syncthreads();
        return;  // no partial row: the finishing blocks' bounded polls run out as well
    }

    // Partial row: (hi, lo) for each column, two columns per 16-byte store; plain sums four
    // columns per 16-byte store when the sums are not compensated.
    const int P = gridDim.x;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = v * nthreads + tid;
        if (vi < nvec) {
            if constexpr (KAHAN) {
                float2* pg = a.part + (size_t)blockIdx.x * cols + (size_t)vi * V;
                float2* pb = a.part + ((size_t)P + blockIdx.x) * cols + (size_t)vi * V;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    st_part4(pg + 2 * h, f2_lo(sg[v][h]), -f2_lo(cg[v][h]), f2_hi(sg[v][h]), -f2_hi(cg[v][h]));
                    if constexpr (!RMS)
                        st_part4(pb + 2 * h, f2_lo(sb[v][h]), -f2_lo(cb[v][h]), f2_hi(sb[v][h]), -f2_hi(cb[v][h]));
                }
            } else {
                float* pg = reinterpret_cast<float*>(a.part) + (size_t)blockIdx.x * cols + (size_t)vi * V;
                float* pb = reinterpret_cast<float*>(a.part) + ((size_t)P + blockIdx.x) * cols + (size_t)vi * V;
#pragma unroll
                for (int h = 0; h < H; h += 2) {
                    st_part4(pg + 2 * h, f2_lo(sg[v][h]), f2_hi(sg[v][h]), f2_lo(sg[v][h + 1]), f2_hi(sg[v][h + 1]));
                    if constexpr (!RMS)
                        st_part4(pb + 2 * h, f2_lo(sb[v][h]), f2_hi(sb[v][h]), f2_lo(sb[v][h + 1]), f2_hi(sb[v][h + 1]));
                }
            }
        }
    }
    finish_if_owner<T>(a, reinterpret_cast<float*>(smem_raw));
}

// ---------------------------------------------------------------------------------------
// Scalar kernel (any alignment, any width).  Each column is owned by one thread of the
// block; its compensated running sums live in shared memory when 16 bytes per column fit,
// else in a region of the workspace behind the partial rows (L2-resident), so that the
// partial rows themselves are written only once, when they are final.
// ---------------------------------------------------------------------------------------
template <typename T, bool RMS>
__global__ void __launch_bounds__(kBwdScalarThreads, 1) bwd_scalar_kernel(const KParams a) {
    using IO = Io<T>;
    pdl_enter();
    constexpr int NW = kBwdScalarThreads / 32;
    extern __shared__ __align__(16) float smem_f[];
    __shared__ float red[2][NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = a.cols, P = gridDim.x;
    const RowDivisor rdiv(cols);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const T* __restrict__ xr = static_cast<const T*>(a.xr);
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    T* __restrict__ dx = static_cast<T*>(a.dx);
    int r0, r1;
    row_range(a.rows, r0, r1);
    // acc_g[c] = (s, c) Kahan pair of dgamma, acc_b[c] the one of dbeta.
    const bool in_smem = a.stages != 0;  // the host sets it when 16 * cols bytes fit
    float2* acc_g = in_smem ? reinterpret_cast<float2*>(smem_f)
                            : a.acc + (size_t)blockIdx.x * cols;
    float2* acc_b = in_smem ? reinterpret_cast<float2*>(smem_f) + cols
                            : a.acc + ((size_t)P + blockIdx.x) * cols;
    for (int j = tid; j < cols; j += kBwdScalarThreads)
        acc_g[j] = acc_b[j] = make_float2(0.f, 0.f);

    for (int row = r0; row < r1; ++row) {
        const size_t base = (size_t)row * cols;
        const float mu = RMS ? 0.f : a.mean[row], rs = a.rstd[row];  // RMSNorm: no mean
        float sg = 0.f, sgx = 0.f;
        for (int j = tid; j < cols; j += kBwdScalarThreads) {
            const float d = IO::to_f(dy[base + j]);
            const float xh = (IO::to_f(xr[base + j]) - mu) * rs;
            const float g = __fmul_rn(IO::to_f(gamma[j]), d);
            sg += g;
            sgx += g * xh;
            float2 pg = acc_g[j];
            kahan_add(pg.x, pg.y, __fmul_rn(d, xh));
            acc_g[j] = pg;
            if constexpr (!RMS) {
                float2 pb = acc_b[j];
                kahan_add(pb.x, pb.y, d);
                acc_b[j] = pb;
            }
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
        const float mg = RMS ? 0.f : rdiv.div(tg), mgx = rdiv.div(tgx);
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
        st_part2(a.part + (size_t)blockIdx.x * cols + j, pg.x, -pg.y);
        if constexpr (!RMS) st_part2(a.part + ((size_t)P + blockIdx.x) * cols + j, pb.x, -pb.y);
        if (!in_smem) acc_g[j] = acc_b[j] = make_float2(0.f, 0.f);  // the workspace is left zero
    }
    __syncthreads();  // the shared accumulators become the finish scratch
    finish_if_owner<T>(a, smem_f);
}

// ---------------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------------
// Warp path: up to 8 vectors per lane for fp32 (1024 columns), 5 for bf16 (1280 columns),
// 4 for bf16 with compensated sums: beyond that the register-resident column sums no
// longer fit without spilling.
template <typename T, bool K, bool RMS>
const void* warp_kernel_k(int vpl) {
    switch (vpl) {
        case 1: return (const void*)bwd_tile_kernel<T, 1, K, RMS>;
        case 2: return (const void*)bwd_tile_kernel<T, 2, K, RMS>;
        case 3: return (const void*)bwd_tile_kernel<T, 3, K, RMS>;
        case 4: return (const void*)bwd_tile_kernel<T, 4, K, RMS>;
        default: break;
    }
    if constexpr (Io<T>::kVec == 8) {
        if (vpl == 5 && !K) return (const void*)bwd_tile_kernel<T, 5, false, RMS>;
    } else {
        switch (vpl) {
            case 5: return (const void*)bwd_tile_kernel<T, 5, K, RMS>;
            case 6: return (const void*)bwd_tile_kernel<T, 6, K, RMS>;
            case 7: return (const void*)bwd_tile_kernel<T, 7, K, RMS>;
            case 8: return (const void*)bwd_tile_kernel<T, 8, K, RMS>;
            default: break;
        }
    }
    return nullptr;
}

// Rows wider than one warp's registers: W = 4 warps per row with 3 or 4 vectors per lane,
// or W = 2 with 3 or 4 (bf16) or 5 (compensated sums) -- the shapes tile_shape picks from.
template <typename T, bool K, bool RMS>
const void* group_kernel_k(int vpl, int W) {
    if (W == 2) {
        if constexpr (K) {
            if (vpl == 5) return (const void*)bwd_tile_kernel<T, 5, K, RMS, 2>;
        }
        if constexpr (Io<T>::kVec == 8) {
            if (vpl == 3) return (const void*)bwd_tile_kernel<T, 3, K, RMS, 2>;
            if (vpl == 4) return (const void*)bwd_tile_kernel<T, 4, K, RMS, 2>;
        }
    }
    if constexpr (!K || Io<T>::kVec == 4) {  // (bf16 compensated: one row per tile; not used)
        if (W == 4) return vpl == 3 ? (const void*)bwd_tile_kernel<T, 3, K, RMS, 4>
                         : vpl == 4 ? (const void*)bwd_tile_kernel<T, 4, K, RMS, 4> : nullptr;
    }
    return nullptr;
}

template <typename T, bool RMS>
const void* warp_kernel(int vpl, bool kahan, int W) {
    if (W > 1) {
        if constexpr (Io<T>::kVec == 4)  // fp32 sums are always compensated
            return kahan ? group_kernel_k<T, true, RMS>(vpl, W) : nullptr;
        else
            return kahan ? group_kernel_k<T, true, RMS>(vpl, W) : group_kernel_k<T, false, RMS>(vpl, W);
    }
    return kahan ? warp_kernel_k<T, true, RMS>(vpl) : warp_kernel_k<T, false, RMS>(vpl);
}

int warp_max_vpl(Dtype dt, bool kahan) { return dt == Dtype::F32 ? 8 : (kahan ? 4 : 5); }

// Warps per row of the tile kernel and vectors per lane: one warp while a lane's share of
// the row fits its registers; else, of 2 warps (3 to 5 vectors per lane) and 4 warps (3 or
// 4), the one that keeps the most rows of a tile in flight, then the one with more warps
// (W = 0: the row is too wide, or only one row per tile would fit: the block-per-row kernel
// is used).  Measured on GB300: bf16 8192 x 2560 2 x 5 / 4 x 3 (3 rows per tile each):
// 34.3 / 31.7 us; fp32 8192 x 1280 2 x 5 (5 rows) / 4 x 3 (3 rows): 26.1 / 28.6 us; bf16
// 65600 x 2560, compensated sums: 2 x 5 (3 rows) / 4 x 3 (1 row): 281 / 438 us.
void tile_shape(Dtype dt, int nvec, bool kahan, int* W, int* vpl) {
    *W = 1;
    *vpl = (nvec + 31) / 32;
    if (*vpl <= warp_max_vpl(dt, kahan)) return;
    const int H = dt == Dtype::F32 ? 2 : 4;
    int best_w = 0, best_v = 0, best_rt = 1;
    for (int w = 2; w <= 4; w *= 2) {
        const int v = (nvec + 32 * w - 1) / (32 * w);
        const bool built = w == 4 ? (v == 3 || v == 4) && !(kahan && dt != Dtype::F32)
                                  : (v == 5 ? kahan : (v == 3 || v == 4) && dt != Dtype::F32);
        if (!built) continue;
        const int rt = tile_rows_for(H, v, kahan, w);
        if (rt >= best_rt && rt > 1) {  // ties go to the larger W
            best_w = w;
            best_v = v;
            best_rt = rt;
        }
    }
    *W = best_w;
    *vpl = best_v;
}

// Block path: cols <= 16384 and 512 threads give at most 4 vectors per thread for bf16 and
// 8 for fp32.  Compensated (Kahan) column sums where the plan asks for them: the registers
// are there for at most 16 columns per thread.
template <typename T, bool RMS>
const void* block_kernel(int vpt, bool kahan) {
    if constexpr (Io<T>::kVec == 8) {
        switch (vpt) {
            case 1: return kahan ? (const void*)bwd_block_kernel<T, 1, true, RMS> : (const void*)bwd_block_kernel<T, 1, false, RMS>;
            case 2: return kahan ? (const void*)bwd_block_kernel<T, 2, true, RMS> : (const void*)bwd_block_kernel<T, 2, false, RMS>;
            case 3: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 3, false, RMS>;
            case 4: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 4, false, RMS>;
            default: return nullptr;
        }
    } else {
        switch (vpt) {
            case 1: return kahan ? (const void*)bwd_block_kernel<T, 1, true, RMS> : (const void*)bwd_block_kernel<T, 1, false, RMS>;
            case 2: return kahan ? (const void*)bwd_block_kernel<T, 2, true, RMS> : (const void*)bwd_block_kernel<T, 2, false, RMS>;
            case 3: return kahan ? (const void*)bwd_block_kernel<T, 3, true, RMS> : (const void*)bwd_block_kernel<T, 3, false, RMS>;
            case 4: return kahan ? (const void*)bwd_block_kernel<T, 4, true, RMS> : (const void*)bwd_block_kernel<T, 4, false, RMS>;
            case 5: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 5, false, RMS>;
            case 6: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 6, false, RMS>;
            case 7: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 7, false, RMS>;
            case 8: return kahan ? nullptr : (const void*)bwd_block_kernel<T, 8, false, RMS>;
            default: return nullptr;
        }
    }
}

template <bool RMS>
const void* kernel_for(Dtype dt, const BwdPlan& p) {
    const bool f = dt == Dtype::F32;
    if (p.path == kPathWarp)
        return f ? warp_kernel<float, RMS>(p.per_thread, p.kahan, p.wpr)
                 : warp_kernel<__nv_bfloat16, RMS>(p.per_thread, p.kahan, p.wpr);
    if (p.path == kPathBlock)
        return f ? block_kernel<float, RMS>(p.per_thread, p.kahan)
                 : block_kernel<__nv_bfloat16, RMS>(p.per_thread, p.kahan);
    return f ? (const void*)bwd_scalar_kernel<float, RMS>
             : (const void*)bwd_scalar_kernel<__nv_bfloat16, RMS>;
}


template <bool RMS>
cudaError_t plan_bwd_t(Dtype dt, int rows, int cols, bool aligned, int path_override,
                       BwdPlan* plan) {
    const DeviceInfo& di = device_info(-1);
    const int V = dt == Dtype::F32 ? 4 : 8;
    const int esize = dt == Dtype::F32 ? 4 : 2;
    BwdPlan p;
    p.rms = RMS;
    if (aligned && path_override != kPathScalar) {
        const int nvec = cols / V;
        // The warp path keeps each lane's column sums over all the rows its warp handles:
        // compensated for fp32 I/O, and for bf16 once those chains can get long.
        const bool wk = dt == Dtype::F32 || rows > kWarpPathMaxRows;
        int W, vpl;
        tile_shape(dt, nvec, wk, &W, &vpl);
        const bool warp_fits = W > 0;
        if (warp_fits && (path_override == kPathWarp || path_override == kPathAuto)) {
            p.path = kPathWarp;
            p.per_thread = vpl;
            p.wpr = W;
            p.tile_rows = tile_rows_for(dt == Dtype::F32 ? 2 : 4, vpl, wk, W);
            p.threads = (p.tile_rows * W + 1) * 32;
            p.kahan = wk;
            const size_t slot = 2ull * p.tile_rows * cols * esize;  // a tile of dy and of x
            const size_t combine = (wk ? 4ull : 2ull) * p.tile_rows * cols * 4;
            // About four tiles in flight per SM, split over the blocks the registers allow
            // on an SM, within each block's share of its shared memory.  Measured on GB300:
            // deeper rings request a block's whole share of rows at once, the DRAM queue then
            // serves blocks roughly in launch order and the late ones set the kernel's end
            // (bf16 8192x768, two blocks per SM: 5 stages 14.2 us, 2 stages 13.5 us; bf16
            // 8192x1280, one block per SM: 6 stages 18.8 us, 4 stages 18.5 us, 2 stages 19.4 us).
            // With W > 1 warps per row, 3 tiles (bf16 8192x3072: 2 / 3 / 4 / 6 stages
            // 34.0 / 32.6 / 33.1 / 34.8 us).
            const void* kern = kernel_for<RMS>(dt, p);
            if (!kern) return cudaErrorInvalidValue;
            const int occ_regs = std::max(1, blocks_per_sm(kern, p.threads, 0));
            const size_t share = std::min<size_t>(
                (size_t)di.smem_optin, (size_t)di.smem_per_sm / occ_regs - 1024);
            int stages = (int)std::min<size_t>(std::min(kMaxStages, W > 1 ? 3 : 4 / occ_regs), share / slot);
            stages = std::max(2, stages);
            p.stages = stages;
            // The ring, reused afterwards for the warps' sums.
            p.smem = std::max<size_t>({(size_t)stages * slot, combine, (size_t)p.threads * 32});
        } else {
            p.path = kPathBlock;
            p.per_thread = (nvec + kBwdBlockMaxThreads - 1) / kBwdBlockMaxThreads;
            const int t = (nvec + p.per_thread - 1) / p.per_thread;
            p.threads = std::max(32, (t + 31) / 32 * 32);
            // Compensated column sums: always for fp32 I/O (as far as the registers go); for
            // bf16 only when a thread's chain of rows can be long (more than 64 rows per
            // block even at one block per SM): over short chains an fp32 sum is far more
            // accurate than the bf16 result it is rounded to.
            p.kahan = dt == Dtype::F32 ? p.per_thread <= 4
                                       : (p.per_thread <= 2 && rows > 64 * di.sms);
            const size_t slot = 2ull * cols * esize;  // a row of dy and of x
            const void* kern = kernel_for<RMS>(dt, p);
            if (!kern) return cudaErrorInvalidValue;
            const int occ_regs = std::max(1, blocks_per_sm(kern, p.threads, 0));
            const size_t share = std::min<size_t>(
                (size_t)di.smem_optin, (size_t)di.smem_per_sm / occ_regs - 1024);
            // Rows in flight: up to 3, within the block's share of shared memory.  Measured on
            // GB300 at bf16 4096 x 8192: 2 / 3 / 4 rows 45.0 / 41.7 / 42.5 us; refilling a slot
            // a pass earlier than after the row's last use (more lead) took 60.7 us -- deeper
            // prefetch delays every block's first rows in the DRAM queue.
            const int stages = (int)std::min<size_t>(kBlockStages, share / slot);
            p.stages = std::max(1, stages);
            p.smem = std::max<size_t>((size_t)p.stages * slot, (size_t)p.threads * 32);
        }
    }
    if (p.path == kPathAuto) {
        p.path = kPathScalar;
        p.threads = kBwdScalarThreads;
        const size_t acc = 16ull * cols;  // (hi, lo) pairs for both statistics
        const bool fits = bwd_scalar_acc_in_smem(cols, (size_t)di.smem_optin);
        p.smem = std::max<size_t>(fits ? acc : 0, (size_t)kBwdScalarThreads * 16);
        p.stages = fits ? 1 : 0;  // tells the kernel where its accumulators live
    }
    if (p.smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
    const void* kern = kernel_for<RMS>(dt, p);
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    const int occ = blocks_per_sm(kern, p.threads, p.smem);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int need = p.path == kPathWarp ? (rows + p.tile_rows - 1) / p.tile_rows : rows;
    p.grid = std::max(1, std::min(need, di.sms * occ));
    *plan = p;
    return cudaSuccess;
}

template <bool RMS>
cudaError_t launch_bwd_t(Dtype dt, const BwdArgs& a, const BwdPlan& p, cudaStream_t stream,
                         int* launches) {
    *launches = 0;
    const void* kern = kernel_for<RMS>(dt, p);
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
    k.acc = bwd_plan_acc_region(p) ? k.part + 2ull * (size_t)p.grid * (size_t)a.cols : nullptr;
    k.compact = (p.path == kPathScalar || p.kahan) ? 0 : 1;
    k.nstat = RMS ? 1 : 2;
    k.P = p.grid;
    // The block-per-row kernel hands the finish to a separate dependent launch: there every
    // block would finish (one block per SM, wide rows) and the early ones poll rows not yet
    // written.  Measured on GB300: bf16 4096 x 8192 backward 41.8 -> 40.9 us split; the warp
    // kernel's in-kernel finish is faster (bf16 8192 x 768 12.0 us against 13.3 split).
    const bool split = p.path == kPathBlock;
    k.split_finish = split ? 1 : 0;
    {
        const int U = k.compact ? (a.cols % 4 == 0 ? 4 : a.cols % 2 == 0 ? 2 : 1)
                                : (a.cols % 2 == 0 ? 2 : 1);
        const int nw = (split ? kFinThreads : p.threads) / 32;
        k.fin_rw = fin_warps_per_group(nw, p.grid, (k.compact ? 1 : 2) * U);
    }
    k.ctr = a.counters;
    k.status = a.status;
    k.limit_ns = a.wait_limit_ns;
    k.wait_extra = a.wait_extra;
    k.stages = p.stages;
    void* args[] = {&k};
    if (split) {
        cudaError_t e = launch_kernel(kern, dim3(p.grid), dim3(p.threads), p.smem, stream, args, false);
        if (e != cudaSuccess) return e;
        const int U = k.compact ? (a.cols % 4 == 0 ? 4 : a.cols % 2 == 0 ? 2 : 1)
                                : (a.cols % 2 == 0 ? 2 : 1);
        const int ng = (k.nstat * (a.cols / U) + kFinUnits - 1) / kFinUnits;
        const void* fk = dt == Dtype::F32 ? (const void*)bwd_finish_kernel<float>
                                          : (const void*)bwd_finish_kernel<__nv_bfloat16>;
        e = launch_kernel(fk, dim3(std::max(1, ng)), dim3(kFinThreads), 0, stream, args, false);
        if (e == cudaSuccess) *launches = 2;
        return e;
    }
    // A cooperative launch: all blocks co-resident, as the finish's polls need.
    cudaError_t e = launch_kernel(kern, dim3(p.grid), dim3(p.threads), p.smem, stream, args, true);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace
}  // namespace lnk
