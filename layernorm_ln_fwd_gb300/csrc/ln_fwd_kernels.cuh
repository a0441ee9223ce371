// ln_fwd_kernels.cuh -- forward kernels of the fused residual-add + LayerNorm and, with
// RMS = true, of the fused residual-add + RMSNorm, and their launch planning.  Included by
// ln_fwd.cu (LayerNorm instantiations) and rms_fwd.cu (RMSNorm instantiations), so that the
// two sets compile in parallel.
//
// For each row: s = x + res (fp32), stored as res_out after rounding to the I/O type; the
// row statistics of the stored values; then
//   LayerNorm: out = gamma * (s - mu) * rstd + beta, rstd = 1 / sqrt(var + eps)
//              ("Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1;
//              residual fusion as in "llm.c: the llmc/ CUDA kernel layer", section 3.2);
//   RMSNorm:   out = gamma * s * r, r = 1 / sqrt(mean(s^2) + eps) ("GPU Performance from
//              First Principles", section 6.1, the fused add + RMSNorm), r stored in `rstd`.
//
// LayerNorm statistics in one reduction, without the cancellation of E[s^2] - E[s]^2 that
// breaks rows whose mean dwarfs their spread ("Accelerating Transformer on GPU (I)", section
// 4.2): shifted sums.  With d = s - K for K = the row's first stored value, sum d and sum d^2
// are reduced together (one xor butterfly, plus one cross-warp exchange for a block per row)
// and var = sum d^2 / n - (sum d / n)^2.  Since sum d^2 / n = var + (mean - K)^2 this keeps
// all but log2(1 + (mean - K)^2 / var) bits, a few when K lies within a few standard
// deviations of the mean, as a value of the row almost always does.  When it does not --
// (mean - K)^2 > 16 var, an outlier in the first column, say -- the row is summed a second
// time about K' = K + mean(d), which lies within rounding of the mean, and the two sums
// then give the variance and the small correction of K' (the corrected two-pass algorithm):
// full precision whatever the first value is, at the price of a second reduction for those
// rows only.  xhat = (s - K) * rstd - mean(d) * rstd (one fma); the mean is stored as
// K + mean(d) and rstd = rsqrtf(var + eps), both in fp32.  The scalar kernel keeps Welford
// summaries per thread and merges them pairwise (Welford/Chan, same section).
//
// Three kernel families compute the same function:
//  * warp per row (rows of at most 256 vectors of 16 bytes): tiles of 7 rows are staged in
//    shared memory by bulk copies several tiles ahead; each warp normalises one row with
//    128-bit reads and stores and one xor butterfly, no block barrier; bf16 rows of 257-384
//    vectors take 4 warps per row (tiles of 3 rows), which add their sums through shared
//    memory announced on an mbarrier;
//  * block per row (wider rows): a persistent block streams rows into shared memory with
//    bulk copies (cp.async.bulk, completed on an mbarrier) several rows ahead, so each row
//    is read from HBM once; one warp butterfly plus one cross-warp exchange per row;
//  * scalar block per row, for rows that are not 16-byte multiples or unaligned pointers.
#pragma once

#include <algorithm>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

// Consumer warps = rows per tile, plus one producer warp: 8 warps, because registers are
// allocated to warps in groups of four (a 9-warp block would pay for 12).
constexpr int kTileRows = 7;
constexpr int kTileThreads = (kTileRows + 1) * 32;
// Rows per tile with W > 1 warps per row (bf16, VPL vectors per lane): one block per SM of
// as many warps as the registers allow -- a thread keeps gamma, beta, the row's values and
// their shifted pairs (~28 registers per vector) plus ~32 -- paid for in fours.
__host__ __device__ constexpr int fwd_tile_rows(int vpl, int W) {
    if (W == 1) return kTileRows;
    const int regs = 28 * vpl + 32;
    const int warps = (65536 / (32 * ((regs + 7) / 8 * 8))) / 4 * 4;
    return (warps - 1) / W;
}
__host__ __device__ constexpr int fwd_tile_threads(int vpl, int W) {
    return (fwd_tile_rows(vpl, W) * W + 1) * 32;
}
constexpr int kFwdBlockMaxThreads = 512;
constexpr int kFwdScalarThreads = 256;
constexpr int kMaxStages = 4;

// The shifted sums leave too few bits once (mean - K)^2 exceeds this many variances.
constexpr float kShiftLimit = 16.f;

// One xor butterfly of a single value over the warp (the same bits in every lane).
__device__ __forceinline__ float warp_sum1(float a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(kFullMask, a, o);
    return a;
}

// The prologue of one 16-byte vector: s = res + keep * (x + bias) * scale for the V elements
// starting at element index i0 (a multiple of 4), rounded to the I/O type.  Dropped elements
// take res itself.  kb returns the V keep decisions as bits (bit k: element i0 + k).
template <typename T>
__device__ __forceinline__ uint4 prologue_vec(const uint4& xv, const uint4& rv, const uint4& bv,
                                              const DropoutRng& rng, float scale,
                                              unsigned long long i0, unsigned& kb) {
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 hv[H], r2[H], bias[H], o[H];
    PR::unpack(xv, hv);
    PR::unpack(rv, r2);
    PR::unpack(bv, bias);
    // The generator's words for the vector's 2 H elements (i0 % (2 H) == 0).
    uint32_t w[2 * H];
    const uint4 wa = rng.words(i0 >> 2);
    w[0] = wa.x; w[1] = wa.y; w[2] = wa.z; w[3] = wa.w;
    if constexpr (H == 4) {
        const uint4 wb = rng.words((i0 >> 2) + 1);
        w[4] = wb.x; w[5] = wb.y; w[6] = wb.z; w[7] = wb.w;
    }
    const f2 sc = f2_splat(scale);
    kb = 0;
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const bool k0 = w[2 * h] >= rng.thr, k1 = w[2 * h + 1] >= rng.thr;
        kb |= (k0 ? 1u : 0u) << (2 * h) | (k1 ? 1u : 0u) << (2 * h + 1);
        const f2 t = f2_mul(f2_add(hv[h], bias[h]), sc);
        const f2 kt = f2_make(k0 ? f2_lo(t) : 0.f, k1 ? f2_hi(t) : 0.f);
        o[h] = f2_add(r2[h], kt);
    }
    return PR::pack(o);
}

// Stores vector vi's keep bits kb (0 for a lane past the row's end) in the prologue's bit
// mask: one byte per 8 columns, rows padded to whole bytes.  An fp32 vector holds 4 columns,
// half a byte: the even lane of each pair of lanes (vectors vi and vi + 1, which adjacent
// lanes hold) writes both halves.  Every lane of the warp calls it (the exchange is a
// shuffle).
template <typename T>
__device__ __forceinline__ void store_keep_bits(const Prologue& pro, int row, int vi, bool valid,
                                                unsigned kb) {
    uint8_t* dst = pro.keep_out + (size_t)row * pro.keep_stride;
    if constexpr (Io<T>::kVec == 8) {
        if (valid) dst[vi] = (uint8_t)kb;
    } else {
        const unsigned hi = __shfl_xor_sync(kFullMask, kb, 1);
        if (valid && (vi & 1) == 0) dst[vi >> 1] = (uint8_t)(kb | (hi << 4));
    }
}

// ---------------------------------------------------------------------------------------
// Warp per row, fed by a bulk-copy (TMA) pipeline.
//
// A block has kTileRows (7) consumer warps and one producer warp (with W > 1 warps per row:
// RT rows of W warps each).  A tile is kTileRows (RT) consecutive rows -- one contiguous
// stretch of memory per tensor -- so the producer's lane 0
// fetches a whole tile of x (and of res) with one cp.async.bulk each, `stages` tiles ahead,
// into a ring of shared-memory slots.  Each consumer warp normalises one row of the tile
// from shared memory (128-bit reads, lane l holds vectors l, l+32, ...), writes res_out and
// out with 128-bit streaming stores, and releases the slot.  The full barrier of a slot
// completes when its copies land; the empty barrier when all consumer warps are done.
// The bytes in flight per SM are set by the ring, not by the registers of resident warps.
// ---------------------------------------------------------------------------------------
template <typename T, int VPL, bool HAS_RES, bool RMS, int PRO = 0, int W = 1>
__global__ void __launch_bounds__(fwd_tile_threads(VPL, W), W == 1 && VPL <= (PRO ? 3 : 4) ? 2 : 1)
    fwd_tile_kernel(const T* __restrict__ x, const T* __restrict__ res,
                    const T* __restrict__ gamma, const T* __restrict__ beta, float eps, int rows,
                    int cols, T* __restrict__ out, T* __restrict__ res_out,
                    float* __restrict__ mean, float* __restrict__ rstd, int stages,
                    unsigned* status, uint64_t wait_limit_ns, Prologue pro) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    // RT rows per tile, W warps per row: consumer warp c normalises row c / W of every tile,
    // its lanes taking the vectors (v * W + c % W) * 32 + lane.  With W > 1 the W warps of a
    // row exchange their sums through xval, announced on xbar (one mbarrier per row of the
    // tile, double-buffered by exchange parity), and add them in warp order.
    constexpr int RT = fwd_tile_rows(VPL, W);
    constexpr int NCW = RT * W;  // consumer warps; warp NCW is the producer
    constexpr int VSTRIDE = 32 * W;
    static_assert(W == 1 || PRO == 0, "the prologue runs with one warp per row");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    __shared__ uint64_t xbar[W > 1 ? 2 * RT : 1];
    __shared__ float2 xval[W > 1 ? 2 * RT * W : 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wrow = warp / W, wpos = warp - wrow * W;
    const int lane_vec = wpos * 32 + lane;
    const int nvec = cols / V;
    const RowDivisor rdiv(cols);
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned tile_bytes = (unsigned)RT * row_bytes;
    const unsigned slot_bytes = (HAS_RES ? 2u : 1u) * tile_bytes;
    const int ntiles = (rows + RT - 1) / RT;
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
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

    if (warp == NCW) {  // producer
        if (lane == 0) {
            int k = 0;
            RingPos pos;
            for (; k < my_tiles; ++k, pos.next(stages)) {
                const int slot = pos.slot;
                // A slot's second and later fills wait for the consumers of the previous pass.
                if (k >= stages && !mbar_wait(&empty_bar[slot], pos.phase ^ 1u, wait_limit_ns)) {
                    raise_status(status, kStatusTimeout);
                    break;
                }
                const int r0 = ((int)blockIdx.x + k * (int)gridDim.x) * RT;
                const unsigned bytes = (unsigned)min(RT, rows - r0) * row_bytes;
                unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
                mbar_arrive_expect_tx(&full_bar[slot], (HAS_RES ? 2u : 1u) * bytes);
                bulk_g2s(dst, x + (size_t)r0 * cols, bytes, &full_bar[slot]);
                if (HAS_RES) bulk_g2s(dst + tile_bytes, res + (size_t)r0 * cols, bytes, &full_bar[slot]);
            }
            // Every copy issued has landed before this block's shared memory is released.
            for (int j = max(0, k - stages); j < k; ++j)
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, wait_limit_ns);
        }
        return;
    }

    // Consumers: gamma (and beta) of this lane's columns, as fp32 pairs, for every row.
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 gp[VPL][H], bp[VPL][H];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        const int vi = v * VSTRIDE + lane_vec;
        PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gp[v]);
        if constexpr (!RMS)
            PR::unpack(vi < nvec ? ld_keep(beta + (size_t)vi * V) : make_uint4(0, 0, 0, 0), bp[v]);
    }
    // The prologue's bias (read through L1 where it is used) and generator.
    const T* bptr = static_cast<const T*>(pro.bias);
    const DropoutRng& rng = pro.rng;
    const bool write_res = res_out != nullptr;
    // W > 1: the row's W warps add their sums (a, b) in warp order; every warp gets the same
    // bits.  `xok` turns false when a partner's sums did not arrive within the time limit.
    int xstep = 0;
    bool xok = true;
    auto row_total = [&](float& a, float& b) {
        if constexpr (W > 1) {
            const int xi = (xstep & 1) * RT + wrow;
            if (lane == 0) {
                xval[xi * W + wpos] = make_float2(a, b);
                mbar_arrive(&xbar[xi]);
            }
            xok = __all_sync(kFullMask, mbar_wait(&xbar[xi], (unsigned)(xstep >> 1) & 1u, wait_limit_ns)) && xok;
            ++xstep;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const float2 q = xval[xi * W + j];
                s0 += q.x;
                s1 += q.y;
            }
            a = s0;
            b = s1;
        }
    };
    RingPos pos;
    for (int k = 0; k < my_tiles; ++k, pos.next(stages)) {
        const int slot = pos.slot;
        const bool ok = mbar_wait(&full_bar[slot], pos.phase, wait_limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            if (lane == 0) raise_status(status, kStatusTimeout);
            break;
        }
        const int row = ((int)blockIdx.x + k * (int)gridDim.x) * RT + wrow;
        if (row < rows) {
            const size_t base = (size_t)row * cols;
            const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes +
                                                     (size_t)wrow * row_bytes);
            const T* rsm = xs + (size_t)RT * cols;
            // s = x + res, rounded to the stored type (one packed add per pair for bf16), or
            // the prologue's res + keep * (x + bias) * scale; it is what gets normalised.
            auto s_vec_kb = [&](int v, unsigned& kb) {
                const int vi = v * VSTRIDE + lane_vec;
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)vi * V);
                if constexpr (PRO)
                    return prologue_vec<T>(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V),
                                           ld_keep(bptr + (size_t)vi * V), rng, pro.scale,
                                           base + (size_t)vi * V, kb);
                else
                    return HAS_RES ? IO::add_round(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V))
                                   : xv;
            };
            auto s_vec = [&](int v) {
                unsigned kb;
                return s_vec_kb(v, kb);
            };
            uint4 sp[VPL];
            unsigned kbv[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * VSTRIDE + lane_vec;
                kbv[v] = 0;
                if (vi < nvec) {
                    sp[v] = s_vec_kb(v, kbv[v]);
                    if (write_res) st_stream(res_out + base + (size_t)vi * V, sp[v]);
                } else {
                    sp[v] = make_uint4(0, 0, 0, 0);
                }
            }
            if constexpr (PRO == 2) {
#pragma unroll
                for (int v = 0; v < VPL; ++v)
                    store_keep_bits<T>(pro, row, v * 32 + lane, v * 32 + lane < nvec, kbv[v]);
            }
            if constexpr (RMS) {
                // Sum of squares (the low halves of the pairs take the even columns, the high
                // halves the odd ones; two accumulators halve the dependent chain).
                f2 sv[VPL][H];
                f2 q[2] = {f2_splat(0.f), f2_splat(0.f)};
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    PR::unpack(sp[v], sv[v]);
                    if (v * VSTRIDE + lane_vec < nvec) {
#pragma unroll
                        for (int h = 0; h < H; ++h) q[h & 1] = f2_fma(sv[v][h], sv[v][h], q[h & 1]);
                    }
                }
                const f2 q2 = f2_add(q[0], q[1]);
                float ss = warp_sum1(f2_lo(q2) + f2_hi(q2));  // the one reduction
                float unused = 0.f;
                row_total(ss, unused);
                const float r = rsqrtf(rdiv.div(ss) + eps);
                if (lane == 0 && wpos == 0) rstd[row] = r;
                const f2 r2 = f2_splat(r);
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const int vi = v * VSTRIDE + lane_vec;
                    if (vi < nvec) {
                        f2 o[H];
#pragma unroll
                        for (int h = 0; h < H; ++h) o[h] = f2_mul(gp[v][h], f2_mul(sv[v][h], r2));
                        st_stream(out + base + (size_t)vi * V, PR::pack(o));
                    }
                }
            } else {
                // Shifted sums: K = the row's first stored value (lane 0's; with W > 1 each
                // warp forms it from the row in shared memory).  The low halves of the pairs
                // sum the even columns, the high halves the odd ones.
                float K;
                if constexpr (W == 1) {
                    K = __shfl_sync(kFullMask, first_value<T>(sp[0]), 0);
                } else {
                    const uint4 x0 = *reinterpret_cast<const uint4*>(xs);
                    K = first_value<T>(HAS_RES ? IO::add_round(x0, *reinterpret_cast<const uint4*>(rsm)) : x0);
                }
                f2 d[VPL][H];
                float md, var;
                auto shifted_sums = [&](auto s_of, float sd_shift) {
                    const f2 K2 = f2_splat(sd_shift);
                    f2 a = f2_splat(0.f), q = f2_splat(0.f);
#pragma unroll
                    for (int v = 0; v < VPL; ++v) {
                        if (v * VSTRIDE + lane_vec < nvec) {
                            PR::unpack(s_of(v), d[v]);
#pragma unroll
                            for (int h = 0; h < H; ++h) {
                                d[v][h] = f2_sub(d[v][h], K2);
                                a = f2_add(a, d[v][h]);
                                q = f2_fma(d[v][h], d[v][h], q);
                            }
                        }
                    }
                    float sd = f2_lo(a) + f2_hi(a), sd2 = f2_lo(q) + f2_hi(q);
                    warp_sum2(sd, sd2);
                    row_total(sd, sd2);
                    md = rdiv.div(sd);
                    var = rdiv.div(sd2) - md * md;
                };
                shifted_sums([&](int v) { return sp[v]; }, K);  // the one reduction of the row
                if (md * md > kShiftLimit * var) {
                    // K is far from the mean (warp-uniform: every lane has the same sums): a
                    // second reduction about K + mean(d), on s re-read from shared memory.
                    K += md;
                    shifted_sums(s_vec, K);
                }
                const float rs = rsqrtf(fmaxf(var, 0.f) + eps);
                if (lane == 0 && wpos == 0) {
                    mean[row] = K + md;
                    rstd[row] = rs;
                }
                // out = gamma * ((s - K) * rs - md * rs) + beta
                const f2 rs2 = f2_splat(rs), nmr2 = f2_splat(-md * rs);
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const int vi = v * VSTRIDE + lane_vec;
                    if (vi < nvec) {
                        f2 o[H];
#pragma unroll
                        for (int h = 0; h < H; ++h)
                            o[h] = f2_fma(gp[v][h], f2_fma(d[v][h], rs2, nmr2), bp[v][h]);
                        st_stream(out + base + (size_t)vi * V, PR::pack(o));
                    }
                }
            }
        }
        if (!xok) {  // (W > 1) a warp of this row stopped: stop too, bounded
            if (lane == 0) raise_status(status, kStatusTimeout);
            break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp is done with the slot
    }
}

// ---------------------------------------------------------------------------------------
// Block per row with bulk-copy staging.
//
// Shared memory: `stages` slots, each holding the row of x and (if present) the row of res;
// one mbarrier per slot.  Thread 0 keeps `stages` rows in flight: after a row is consumed
// (end-of-row barrier) it refills that slot with the row `stages` iterations ahead.
// Thread t of the block owns vectors t, t + blockDim.x, ... of every row.
// ---------------------------------------------------------------------------------------
template <typename T, int VPT, bool HAS_RES, bool RMS, int PRO = 0>
__global__ void __launch_bounds__(kFwdBlockMaxThreads, 1)
    fwd_block_kernel(const T* __restrict__ x, const T* __restrict__ res,
                     const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                     int rows, int cols, T* __restrict__ out, T* __restrict__ res_out,
                     float* __restrict__ mean, float* __restrict__ rstd, int stages,
                     unsigned* status, uint64_t wait_limit_ns, Prologue pro) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages];
    __shared__ float red[2][2][32];  // [exchange][sum][warp]: the second one for a re-sum
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nw = nthreads >> 5;
    const int nvec = cols / V;
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned nin = HAS_RES ? 2u : 1u;
    const unsigned slot_bytes = nin * row_bytes;
    const RowDivisor rdiv(cols);

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&full_bar[i], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Set-up done; nothing above touches global memory, so it overlaps the previous grid.
    pdl_enter();

    auto issue = [&](int k, int slot) {  // thread 0 only: fetch the k-th row of this block
        const int row = blockIdx.x + k * gridDim.x;
        if (row >= rows) return;
        unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], slot_bytes);
        bulk_g2s(dst, x + (size_t)row * cols, row_bytes, &full_bar[slot]);
        if (HAS_RES) bulk_g2s(dst + row_bytes, res + (size_t)row * cols, row_bytes, &full_bar[slot]);
    };
    if (tid == 0)
        for (int k = 0; k < stages; ++k) issue(k, k);

    // gamma (and beta) for this thread's vectors (the same columns in every row), as pairs.
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 gp[VPT][H], bp[VPT][H];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = v * nthreads + tid;
        PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gp[v]);
        if constexpr (!RMS)
            PR::unpack(vi < nvec ? ld_keep(beta + (size_t)vi * V) : make_uint4(0, 0, 0, 0), bp[v]);
    }
    // The prologue's bias (read through L1 where it is used) and generator.
    const T* bptr = static_cast<const T*>(pro.bias);
    const DropoutRng& rng = pro.rng;

    // The block's sum of (a, b): one warp butterfly, one exchange through shared memory
    // (exchange `e` of the row), then every thread adds the warps' sums in the same order, so
    // every thread holds the same bits.  Returns false if a copy timed out (abort).
    auto block_sum2 = [&](int e, float& a, float& b) {
        warp_sum2(a, b);
        if (lane == 0) {
            red[e][0][warp] = a;
            red[e][1][warp] = b;
        }
        __syncthreads();
        if (abort_flag) return false;
        sum_warp_values2(red[e][0], red[e][1], nw, a, b);  // the same bits in every thread
        return true;
    };

    const bool write_res = res_out != nullptr;
    int k = 0;
    RingPos pos;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, ++k, pos.next(stages)) {
        const int slot = pos.slot;
        if (!mbar_wait(&full_bar[slot], pos.phase, wait_limit_ns)) abort_flag = 1;
        const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes);
        const T* rsm = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes + row_bytes);
        const size_t base = (size_t)row * cols;
        auto s_vec_kb = [&](int v, unsigned& kb) {
            const int vi = v * nthreads + tid;
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)vi * V);
            if constexpr (PRO)
                return prologue_vec<T>(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V),
                                       ld_keep(bptr + (size_t)vi * V), rng, pro.scale,
                                       base + (size_t)vi * V, kb);
            else
                return HAS_RES ? IO::add_round(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V))
                               : xv;
        };
        auto s_vec = [&](int v) {
            unsigned kb;
            return s_vec_kb(v, kb);
        };

        uint4 sp[VPT];
        unsigned kbv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            kbv[v] = 0;
            if (vi < nvec) {
                sp[v] = s_vec_kb(v, kbv[v]);
                if (write_res) st_stream(res_out + base + (size_t)vi * V, sp[v]);
            } else {
                sp[v] = make_uint4(0, 0, 0, 0);
            }
        }
        if constexpr (PRO == 2) {  // nthreads is a multiple of 32: adjacent lanes, adjacent vectors
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                store_keep_bits<T>(pro, row, v * nthreads + tid, v * nthreads + tid < nvec, kbv[v]);
        }
        if constexpr (RMS) {
            f2 sv[VPT][H];
            f2 q2 = f2_splat(0.f);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                PR::unpack(sp[v], sv[v]);
                if (v * nthreads + tid < nvec) {
#pragma unroll
                    for (int h = 0; h < H; ++h) q2 = f2_fma(sv[v][h], sv[v][h], q2);
                }
            }
            float ss = f2_lo(q2), ss_hi = f2_hi(q2);
            if (!block_sum2(0, ss, ss_hi)) break;  // the one cross-warp exchange of the row
            const float r = rsqrtf(rdiv.div(ss + ss_hi) + eps);
            if (tid == 0) rstd[row] = r;
            const f2 r2 = f2_splat(r);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int vi = v * nthreads + tid;
                if (vi < nvec) {
                    f2 o[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) o[h] = f2_mul(gp[v][h], f2_mul(sv[v][h], r2));
                    st_stream(out + base + (size_t)vi * V, PR::pack(o));
                }
            }
        } else {
            // Shifted sums: K = the row's first stored value (every thread reads it from
            // shared memory).  The low halves of the pairs sum the even columns, the high
            // halves the odd ones.
            // (With the prologue every thread recomputes s of the first vector.)
            unsigned kb0;
            const uint4 first = PRO ? prologue_vec<T>(*reinterpret_cast<const uint4*>(xs),
                                                      *reinterpret_cast<const uint4*>(rsm),
                                                      ld_keep(bptr), rng, pro.scale, base, kb0)
                                : HAS_RES ? IO::add_round(*reinterpret_cast<const uint4*>(xs),
                                                          *reinterpret_cast<const uint4*>(rsm))
                                          : *reinterpret_cast<const uint4*>(xs);
            float K = first_value<T>(first);
            f2 d[VPT][H];
            float md = 0.f, var = 0.f;
            auto shifted_sums = [&](auto s_of, float sd_shift, int e) {
                const f2 K2 = f2_splat(sd_shift);
                f2 a2 = f2_splat(0.f), q2 = f2_splat(0.f);
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    if (v * nthreads + tid < nvec) {
                        PR::unpack(s_of(v), d[v]);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            d[v][h] = f2_sub(d[v][h], K2);
                            a2 = f2_add(a2, d[v][h]);
                            q2 = f2_fma(d[v][h], d[v][h], q2);
                        }
                    }
                }
                float sd = f2_lo(a2) + f2_hi(a2), sd2 = f2_lo(q2) + f2_hi(q2);
                if (!block_sum2(e, sd, sd2)) return false;
                md = rdiv.div(sd);
                var = rdiv.div(sd2) - md * md;
                return true;
            };
            // The one cross-warp exchange of the row.
            if (!shifted_sums([&](int v) { return sp[v]; }, K, 0)) break;
            if (md * md > kShiftLimit * var) {
                // K is far from the mean (block-uniform: every thread has the same sums): a
                // second exchange about K + mean(d), on s re-read from shared memory.
                K += md;
                if (!shifted_sums(s_vec, K, 1)) break;
            }
            const float rs = rsqrtf(fmaxf(var, 0.f) + eps);
            if (tid == 0) {
                mean[row] = K + md;
                rstd[row] = rs;
            }
            // out = gamma * ((s - K) * rs - md * rs) + beta
            const f2 rs2 = f2_splat(rs), nmr2 = f2_splat(-md * rs);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int vi = v * nthreads + tid;
                if (vi < nvec) {
                    f2 o[H];
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = f2_fma(gp[v][h], f2_fma(d[v][h], rs2, nmr2), bp[v][h]);
                    st_stream(out + base + (size_t)vi * V, PR::pack(o));
                }
            }
        }
        __syncthreads();  // the slot and `red` are free again
        if (tid == 0) issue(k + stages, slot);  // row k + stages takes row k's slot
    }

    if (abort_flag) {
        // A copy did not complete in time: record it, then give every issued copy a bounded
        // chance to land before the block's shared memory is released.
        if (tid == 0) {
            raise_status(status, kStatusTimeout);
            for (int j = k; j < k + stages; ++j) {
                const int row = blockIdx.x + j * gridDim.x;
                if (row >= rows) break;
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, wait_limit_ns);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------------
// Scalar block per row: any alignment, any width.  Two passes over global memory (the
// second one hits L1/L2).  LayerNorm: each thread keeps a Welford summary (count, mean and
// M2 of d = s - K, K = the median of five of the row's values) and the summaries are merged
// pairwise (Welford/Chan), with the plain sum of s alongside for the stored mean.  RMSNorm:
// per-thread sums of squares.
// ---------------------------------------------------------------------------------------
template <typename T, bool HAS_RES, bool RMS, int PRO = 0>
__global__ void __launch_bounds__(kFwdScalarThreads)
    fwd_scalar_kernel(const T* __restrict__ x, const T* __restrict__ res,
                      const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                      int rows, int cols, T* __restrict__ out, T* __restrict__ res_out,
                      float* __restrict__ mean, float* __restrict__ rstd, Prologue pro) {
    using IO = Io<T>;
    pdl_enter();
    constexpr int NW = kFwdScalarThreads / 32;
    __shared__ float red[3][NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const RowDivisor rdiv(cols);
    const bool write_res = res_out != nullptr;
    // Counts of values in a row: this thread's (columns tid, tid + 256, ...) and, in lane w,
    // warp w's.  Equal everywhere when cols is a multiple of the block size.
    auto count_of = [&](int t) { return t < cols ? (cols - 1 - t) / kFwdScalarThreads + 1 : 0; };
    const float n_thr = (float)count_of(tid);
    int nw_total = 0;
    for (int j = 0; j < 32 && lane < NW; ++j) nw_total += count_of(lane * 32 + j);
    const float n_warp = (float)nw_total;
    const bool equal = cols % kFwdScalarThreads == 0;
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const size_t base = (size_t)row * cols;
        const DropoutRng& rng = pro.rng;
        auto load_s_k = [&](int j, bool& kept) -> float {
            float v = IO::to_f(x[base + j]);
            kept = true;
            if constexpr (PRO) {
                const float t = (v + IO::to_f(static_cast<const T*>(pro.bias)[j])) * pro.scale;
                kept = rng.keep(base + j);
                return IO::round(IO::to_f(res[base + j]) + (kept ? t : 0.f));
            }
            if (HAS_RES) v = IO::round(v + IO::to_f(res[base + j]));
            return v;
        };
        auto load_s = [&](int j) -> float {
            bool kept;
            return load_s_k(j, kept);
        };
        if constexpr (RMS) {
            float ss = 0.f;
            for (int j = tid; j < cols; j += kFwdScalarThreads) {
                const float sv = load_s(j);
                if (write_res) res_out[base + j] = IO::from_f(sv);
                ss = __fmaf_rn(sv, sv, ss);
            }
            ss = warp_sum1(ss);
            if (lane == 0) red[0][warp] = ss;
            __syncthreads();
            ss = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) ss += red[0][w];
            const float r = rsqrtf(rdiv.div(ss) + eps);
            if (tid == 0) rstd[row] = r;
            for (int j = tid; j < cols; j += kFwdScalarThreads)
                out[base + j] = IO::from_f(IO::to_f(gamma[j]) * (load_s(j) * r));
        } else {
            const float K = PRO ? median5(load_s(sample_col(0, cols)), load_s(sample_col(1, cols)),
                                          load_s(sample_col(2, cols)), load_s(sample_col(3, cols)),
                                          load_s(sample_col(4, cols)))
                                : row_shift<T, HAS_RES>(x + base, HAS_RES ? res + base : nullptr, cols);
            // This thread's summary of its values: their plain sum S, and Welford's running
            // mean and M2 of d = s - K.
            float S = 0.f, md = 0.f, M2 = 0.f, n = 0.f;
            for (int j = tid; j < cols; j += kFwdScalarThreads) {
                bool kept;
                const float sv = load_s_k(j, kept);
                if (write_res) res_out[base + j] = IO::from_f(sv);
                if constexpr (PRO == 2) {  // the warp's 32 columns j0 .. j0 + 31, by ballot
                    const int j0 = j - lane;
                    const unsigned m = cols - j0 >= 32 ? kFullMask : (1u << (cols - j0)) - 1u;
                    const unsigned bits = __ballot_sync(m, kept);
                    if (lane == 0) {
                        uint8_t* dst = pro.keep_out + (size_t)row * pro.keep_stride + j0 / 8;
                        const int nb = min(4, (cols - j0 + 7) / 8);
                        for (int q = 0; q < nb; ++q) dst[q] = (uint8_t)(bits >> (8 * q));
                    }
                }
                S = __fadd_rn(S, sv);
                const float d = __fsub_rn(sv, K);
                n = __fadd_rn(n, 1.f);
                const float delta = __fsub_rn(d, md);
                md = __fadd_rn(md, __fdiv_rn(delta, n));
                M2 = __fmaf_rn(delta, __fsub_rn(d, md), M2);
            }
            if (equal)
                chan_reduce_equal(16, n_thr, S, md, M2);
            else
                chan_reduce_any(n_thr, S, md, M2);
            if (lane == 0) {
                red[0][warp] = S;
                red[1][warp] = md;
                red[2][warp] = M2;
            }
            __syncthreads();
            if (equal) {  // NW = 8 warps of equal counts: lane l takes warp l mod 8
                S = red[0][lane & (NW - 1)];
                md = red[1][lane & (NW - 1)];
                M2 = red[2][lane & (NW - 1)];
                chan_reduce_equal(NW / 2, 32.f * n_thr, S, md, M2);
            } else {
                S = lane < NW ? red[0][lane] : 0.f;
                md = lane < NW ? red[1][lane] : 0.f;
                M2 = lane < NW ? red[2][lane] : 0.f;
                chan_reduce_any(n_warp, S, md, M2);
            }
            const float rs = rsqrtf(rdiv.div(M2) + eps);
            if (tid == 0) {
                mean[row] = rdiv.div(S);
                rstd[row] = rs;
            }
            for (int j = tid; j < cols; j += kFwdScalarThreads) {
                const float sv = load_s(j);
                out[base + j] =
                    IO::from_f(IO::to_f(gamma[j]) * ((sv - K - md) * rs) + IO::to_f(beta[j]));
            }
        }
        __syncthreads();  // `red` is reused by the next row
    }
}

// ---------------------------------------------------------------------------------------
// Host-side dispatch.
// ---------------------------------------------------------------------------------------
// The kernel of a family for a residual (or not); the prologue always has a residual, and
// its instantiations exist only in that form.
template <typename T, int N, bool RMS, int PRO>
const void* tile_ptr(bool has_res) {
    if constexpr (PRO)
        return (const void*)fwd_tile_kernel<T, N, true, RMS, PRO>;
    else
        return has_res ? (const void*)fwd_tile_kernel<T, N, true, RMS, 0>
                       : (const void*)fwd_tile_kernel<T, N, false, RMS, 0>;
}
template <typename T, int N, bool RMS, int PRO>
const void* block_ptr(bool has_res) {
    if constexpr (PRO)
        return (const void*)fwd_block_kernel<T, N, true, RMS, PRO>;
    else
        return has_res ? (const void*)fwd_block_kernel<T, N, true, RMS, 0>
                       : (const void*)fwd_block_kernel<T, N, false, RMS, 0>;
}

// The forward tile kernels with W > 1 warps per row (bf16, no prologue).
template <typename T, int VPL, int W, bool RMS>
const void* wide_ptr(bool has_res) {
    return has_res ? (const void*)fwd_tile_kernel<T, VPL, true, RMS, 0, W>
                   : (const void*)fwd_tile_kernel<T, VPL, false, RMS, 0, W>;
}
template <typename T, bool RMS>
const void* wide_kernel(bool has_res, int W, int vpl) {
    if (W == 4 && vpl == 3) return wide_ptr<T, 3, 4, RMS>(has_res);
    return nullptr;
}

template <bool RMS, int PRO, typename T>
cudaError_t launch_warp(const FwdArgs& a, int vpl, int W, cudaStream_t stream) {
    const void* kern = nullptr;
    const bool has_res = a.res != nullptr;
    const int rt = fwd_tile_rows(vpl, W);
    const int threads = (rt * W + 1) * 32;
#define LNK_FWD_TILE_CASE(N)                                                               \
    case N:                                                                                \
        kern = tile_ptr<T, N, RMS, PRO>(has_res);                                          \
        break;
    if (W > 1) {
        if constexpr (Io<T>::kVec == 8 && PRO == 0)
            kern = wide_kernel<T, RMS>(has_res, W, vpl);
        if (!kern) return cudaErrorInvalidValue;
    } else switch (vpl) {
        LNK_FWD_TILE_CASE(1)
        LNK_FWD_TILE_CASE(2)
        LNK_FWD_TILE_CASE(3)
        LNK_FWD_TILE_CASE(4)
        LNK_FWD_TILE_CASE(5)
        LNK_FWD_TILE_CASE(6)
        LNK_FWD_TILE_CASE(7)
        LNK_FWD_TILE_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
#undef LNK_FWD_TILE_CASE
    const DeviceInfo& di = device_info(-1);
    const size_t slot_bytes = (size_t)(has_res ? 2 : 1) * rt * a.cols * sizeof(T);
    // Two to four tiles in flight per block, two blocks per SM when they fit.
    int stages = (int)std::min<size_t>(kMaxStages, ((size_t)di.smem_optin / 2) / slot_bytes);
    stages = std::max(2, stages);
    const size_t smem = (size_t)stages * slot_bytes;
    if (smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int ntiles = (a.rows + rt - 1) / rt;
    const int occ = std::max(1, blocks_per_sm(kern, threads, smem));
    const int grid = std::max(1, std::min(ntiles, di.sms * occ));
    const T* x = static_cast<const T*>(a.x);
    const T* res = static_cast<const T*>(a.res);
    const T* gamma = static_cast<const T*>(a.gamma);
    const T* beta = static_cast<const T*>(a.beta);
    T* out = static_cast<T*>(a.out);
    T* res_out = static_cast<T*>(a.res_out);
    float eps = a.eps;
    int rows = a.rows, cols = a.cols;
    float* mean = a.mean;
    float* rstd = a.rstd;
    unsigned* status = a.status;
    uint64_t limit = a.wait_limit_ns;
    Prologue pro = a.pro;
    void* args[] = {&x,   &res,     &gamma, &beta, &eps,    &rows,   &cols,
                    &out, &res_out, &mean,  &rstd, &stages, &status, &limit, &pro};
    return launch_kernel(kern, dim3(grid), dim3(threads), smem, stream, args, false);
}

template <bool RMS, int PRO, typename T>
cudaError_t launch_block(const FwdArgs& a, cudaStream_t stream) {
    constexpr int V = Io<T>::kVec;
    const int nvec = a.cols / V;
    // 256 threads per row keep two blocks (two rows being normalised) on an SM; rows too
    // wide for that (more than 4 bf16 or 8 fp32 vectors per thread) take 512 threads.
    constexpr int kMaxVpt = V == 8 ? 4 : 8;
    int vpt = (nvec + 255) / 256;
    if (vpt > kMaxVpt) vpt = (nvec + kFwdBlockMaxThreads - 1) / kFwdBlockMaxThreads;
    const int threads = std::max(32, ((nvec + vpt - 1) / vpt + 31) / 32 * 32);
    const bool has_res = a.res != nullptr;
    const void* kern = nullptr;
#define LNK_FWD_BLOCK_CASE(N)                                                              \
    case N:                                                                                \
        kern = block_ptr<T, N, RMS, PRO>(has_res);                                         \
        break;
    // cols <= 16384: at most 4 vectors per thread for bf16, 8 for fp32.
    if constexpr (V == 8) {
        switch (vpt) {
            LNK_FWD_BLOCK_CASE(1)
            LNK_FWD_BLOCK_CASE(2)
            LNK_FWD_BLOCK_CASE(3)
            LNK_FWD_BLOCK_CASE(4)
            default:
                return cudaErrorInvalidValue;
        }
    } else {
        switch (vpt) {
            LNK_FWD_BLOCK_CASE(1)
            LNK_FWD_BLOCK_CASE(2)
            LNK_FWD_BLOCK_CASE(3)
            LNK_FWD_BLOCK_CASE(4)
            LNK_FWD_BLOCK_CASE(5)
            LNK_FWD_BLOCK_CASE(6)
            LNK_FWD_BLOCK_CASE(7)
            LNK_FWD_BLOCK_CASE(8)
            default:
                return cudaErrorInvalidValue;
        }
    }
#undef LNK_FWD_BLOCK_CASE
    const DeviceInfo& di = device_info(-1);
    const size_t slot_bytes = (size_t)(has_res ? 2 : 1) * a.cols * sizeof(T);
    // Up to kMaxStages rows in flight per block, within about half of an SM's shared memory
    // so that two blocks can share an SM when the rows are small enough.
    const size_t budget = std::max<size_t>(slot_bytes, (size_t)di.smem_optin / 2);
    // About four rows in flight per SM over the blocks the registers allow there (measured
    // on GB300 at 4096x8192 bf16, two blocks per SM: 2 stages 44.4 us, 3 stages 45.0 us).
    const int occ_regs = std::max(1, blocks_per_sm(kern, threads, 0));
    int stages = (int)std::min<size_t>(std::min(kMaxStages, std::max(1, 4 / occ_regs)),
                                       budget / slot_bytes);
    stages = std::max(1, stages);
    const size_t smem = (size_t)stages * slot_bytes;
    if (smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int occ = std::max(1, blocks_per_sm(kern, threads, smem));
    const int grid = std::max(1, std::min(a.rows, di.sms * occ));
    const T* x = static_cast<const T*>(a.x);
    const T* res = static_cast<const T*>(a.res);
    const T* gamma = static_cast<const T*>(a.gamma);
    const T* beta = static_cast<const T*>(a.beta);
    T* out = static_cast<T*>(a.out);
    T* res_out = static_cast<T*>(a.res_out);
    float eps = a.eps;
    int rows = a.rows, cols = a.cols;
    float* mean = a.mean;
    float* rstd = a.rstd;
    unsigned* status = a.status;
    uint64_t limit = a.wait_limit_ns;
    Prologue pro = a.pro;
    void* args[] = {&x,   &res,     &gamma, &beta, &eps,   &rows,   &cols,
                    &out, &res_out, &mean,  &rstd, &stages, &status, &limit, &pro};
    return launch_kernel(kern, dim3(grid), dim3(threads), smem, stream, args, false);
}

template <bool RMS, int PRO, typename T>
cudaError_t launch_scalar(const FwdArgs& a, cudaStream_t stream) {
    const bool has_res = a.res != nullptr;
    const void* kern;
    if constexpr (PRO)
        kern = (const void*)fwd_scalar_kernel<T, true, RMS, PRO>;
    else
        kern = has_res ? (const void*)fwd_scalar_kernel<T, true, RMS, 0>
                       : (const void*)fwd_scalar_kernel<T, false, RMS, 0>;
    const DeviceInfo& di = device_info(-1);
    const int occ = std::max(1, blocks_per_sm(kern, kFwdScalarThreads, 0));
    const int grid = std::max(1, std::min(a.rows, di.sms * occ));
    const T* x = static_cast<const T*>(a.x);
    const T* res = static_cast<const T*>(a.res);
    const T* gamma = static_cast<const T*>(a.gamma);
    const T* beta = static_cast<const T*>(a.beta);
    T* out = static_cast<T*>(a.out);
    T* res_out = static_cast<T*>(a.res_out);
    float eps = a.eps;
    int rows = a.rows, cols = a.cols;
    float* mean = a.mean;
    float* rstd = a.rstd;
    Prologue pro = a.pro;
    void* args[] = {&x, &res, &gamma, &beta, &eps, &rows, &cols, &out, &res_out, &mean, &rstd, &pro};
    return launch_kernel(kern, dim3(grid), dim3(kFwdScalarThreads), 0, stream, args, false);
}

// bf16 rows (no prologue) that take W > 1 warps per row: W and the vectors per lane, or W = 0.
// bf16 rows of 2056-3072 columns: 4 warps per row keep 3 rows of a tile in flight per block,
// where the block-per-row kernel has one per block (8192 x 2560: 32.0 -> 27.4 us, 8192 x 3072
// 39.7 -> 32.8 us on GB300).  Narrower rows stay with one warp per row: at 8192 x 1280 one
// warp 14.7 us, 2 warps x 3 vectors 15.0, 4 x 2 16.3; at 1600 and 2048 columns the shapes
// with 2 or 4 warps per row were within 3 % of one warp.
inline void fwd_wide_shape(int nvec, int* W, int* vpl) {
    *W = 0;
    *vpl = 0;
    if (nvec > 256 && nvec <= 384) {
        *W = 4;
        *vpl = 3;
    }
}

template <bool RMS, int PRO, typename T>
cudaError_t launch_fwd_t(const FwdArgs& a, bool aligned, int path, cudaStream_t stream) {
    constexpr int V = Io<T>::kVec;
    if (!aligned || path == kPathScalar) return launch_scalar<RMS, PRO, T>(a, stream);
    const int nvec = a.cols / V;
    const int vpl = (nvec + 31) / 32;
    if (path == kPathBlock) return launch_block<RMS, PRO, T>(a, stream);
    int W = 0, wv = 0;
    if (V == 8 && PRO == 0) fwd_wide_shape(nvec, &W, &wv);
    if (W > 1) return launch_warp<RMS, PRO, T>(a, wv, W, stream);
    if (vpl <= 8) return launch_warp<RMS, PRO, T>(a, vpl, 1, stream);
    return launch_block<RMS, PRO, T>(a, stream);
}

// The forward of a LayerNorm (RMS = false) or an RMSNorm (RMS = true): one kernel launch.
template <bool RMS, int PRO = 0>
cudaError_t launch_norm_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                            cudaStream_t stream, int* launches) {
    *launches = 0;
    if (a.rows == 0) return cudaSuccess;
    cudaError_t e = dt == Dtype::F32
                        ? launch_fwd_t<RMS, PRO, float>(a, aligned, path_override, stream)
                        : launch_fwd_t<RMS, PRO, __nv_bfloat16>(a, aligned, path_override, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace
}  // namespace lnk
