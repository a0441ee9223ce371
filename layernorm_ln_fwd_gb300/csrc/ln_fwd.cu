// ln_fwd.cu -- forward kernels of the fused residual-add + LayerNorm.
//
// For each row: s = x + res (fp32), stored as res_out after rounding to the I/O type; the
// row statistics of the stored values; out = gamma * (s - mu) * rstd + beta.
// ("Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1; residual
// fusion as in "llm.c: the llmc/ CUDA kernel layer", section 3.2.)
//
// Statistics in one reduction, without the cancellation of E[s^2] - E[s]^2 that breaks rows
// whose mean dwarfs their spread ("Accelerating Transformer on GPU (I)", section 4.2): every
// lane (thread) summarises its own values as (count, mean of d = s - K, M2 of d) -- K is a
// value from the body of the row, so the means are small numbers -- and the summaries
// are merged pairwise with the Welford/Chan update of the same section: one xor butterfly per
// warp, plus one cross-warp exchange and a second butterfly for a block per row.  K is the
// median of five values spread over the row, so it stays in the body of the row whatever a
// few values are.  The merged
// M2 is a sum of non-negative terms, so the variance keeps full precision whichever value K
// is (an outlier in the first column included).  The plain sum of the unshifted values rides
// along in the same butterfly and gives the stored mean; out = gamma * ((d - mean_d) * rstd)
// + beta, and rstd = 1 / sqrt(M2 / n + eps) (rsqrtf), mean and rstd stored in fp32.
//
// Three kernel families compute the same function:
//  * warp per row (rows of at most 256 vectors of 16 bytes): tiles of 7 rows are staged in
//    shared memory by bulk copies several tiles ahead; each warp normalises one row with
//    128-bit reads and stores and one xor butterfly, no block barrier;
//  * block per row (wider rows): a persistent block streams rows into shared memory with
//    bulk copies (cp.async.bulk, completed on an mbarrier) several rows ahead, so each row
//    is read from HBM once; one warp butterfly plus one cross-warp exchange per row;
//  * scalar block per row, for rows that are not 16-byte multiples or unaligned pointers.
#include <algorithm>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

// Consumer warps = rows per tile, plus one producer warp: 8 warps, because registers are
// allocated to warps in groups of four (a 9-warp block would pay for 12).
constexpr int kTileRows = 7;
constexpr int kTileThreads = (kTileRows + 1) * 32;
constexpr int kFwdBlockMaxThreads = 512;
constexpr int kFwdScalarThreads = 256;
constexpr int kMaxStages = 4;

// ---------------------------------------------------------------------------------------
// Warp per row, fed by a bulk-copy (TMA) pipeline.
//
// A block has kTileRows (7) consumer warps and one producer warp.  A tile is kTileRows
// consecutive rows -- one contiguous stretch of memory per tensor -- so the producer's lane 0
// fetches a whole tile of x (and of res) with one cp.async.bulk each, `stages` tiles ahead,
// into a ring of shared-memory slots.  Each consumer warp normalises one row of the tile
// from shared memory (128-bit reads, lane l holds vectors l, l+32, ...), writes res_out and
// out with 128-bit streaming stores, and releases the slot.  The full barrier of a slot
// completes when its copies land; the empty barrier when all consumer warps are done.
// The bytes in flight per SM are set by the ring, not by the registers of resident warps.
// ---------------------------------------------------------------------------------------
template <typename T, int VPL, bool HAS_RES>
__global__ void __launch_bounds__(kTileThreads, VPL <= 4 ? 2 : 1)
    fwd_tile_kernel(const T* __restrict__ x, const T* __restrict__ res,
                    const T* __restrict__ gamma, const T* __restrict__ beta, float eps, int rows,
                    int cols, T* __restrict__ out, T* __restrict__ res_out,
                    float* __restrict__ mean, float* __restrict__ rstd, int stages,
                    unsigned* status, uint64_t wait_limit_ns) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = cols / V;
    const RowDivisor rdiv(cols);
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned tile_bytes = (unsigned)kTileRows * row_bytes;
    const unsigned slot_bytes = (HAS_RES ? 2u : 1u) * tile_bytes;
    const int ntiles = (rows + kTileRows - 1) / kTileRows;
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kTileRows);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // Set-up done; nothing above touches global memory, so it overlaps the previous grid.
    pdl_enter();

    if (warp == kTileRows) {  // producer
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
                const int r0 = ((int)blockIdx.x + k * (int)gridDim.x) * kTileRows;
                const unsigned bytes = (unsigned)min(kTileRows, rows - r0) * row_bytes;
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

    // Consumers: gamma and beta of this lane's columns, as fp32 pairs, for every row.
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 gp[VPL][H], bp[VPL][H];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        const int vi = v * 32 + lane;
        PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gp[v]);
        PR::unpack(vi < nvec ? ld_keep(beta + (size_t)vi * V) : make_uint4(0, 0, 0, 0), bp[v]);
    }
    // This lane's count of values in a row (the same for every row); when the row is a
    // multiple of 32 vectors every lane holds the same count and the butterfly merges equal
    // halves.
    int nv_lane = 0;
#pragma unroll
    for (int v = 0; v < VPL; ++v) nv_lane += v * 32 + lane < nvec ? 1 : 0;
    const float n_lane = (float)(nv_lane * V);
    const float inv_lane = nv_lane ? 1.0f / n_lane : 0.f;
    const bool equal = nvec % 32 == 0;
    // The lanes whose first values make the row's five-value sample for its shift K: spread
    // over the lanes that hold part of the row.
    const int nlanes = min(nvec, 32);
    int sample_lane[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) sample_lane[j] = j * (nlanes - 1) / 4;
    const bool write_res = res_out != nullptr;
    RingPos pos;
    for (int k = 0; k < my_tiles; ++k, pos.next(stages)) {
        const int slot = pos.slot;
        const bool ok = mbar_wait(&full_bar[slot], pos.phase, wait_limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            if (lane == 0) raise_status(status, kStatusTimeout);
            break;
        }
        const int row = ((int)blockIdx.x + k * (int)gridDim.x) * kTileRows + warp;
        if (row < rows) {
            const size_t base = (size_t)row * cols;
            const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes +
                                                     (size_t)warp * row_bytes);
            const T* rsm = xs + (size_t)kTileRows * cols;
            // s = x + res, rounded to the stored type (one packed add per pair for bf16);
            // it is what gets normalised.
            uint4 sp[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * 32 + lane;
                if (vi < nvec) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)vi * V);
                    sp[v] = HAS_RES ? IO::add_round(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V))
                                    : xv;
                    if (write_res) st_stream(res_out + base + (size_t)vi * V, sp[v]);
                } else {
                    sp[v] = make_uint4(0, 0, 0, 0);
                }
            }
            // This lane's summary: the plain sum of s, then d = s - K (K = the median of five
            // of the row's values: the first values of five lanes spread over the row), the
            // mean of d and M2 about it, from registers.  The low halves of the pairs take the
            // even columns, the high halves the odd ones; two accumulators each (even and odd
            // pairs) halve the chains of dependent additions.
            const float f0 = first_value<T>(sp[0]);
            float kv[5];
#pragma unroll
            for (int j = 0; j < 5; ++j) kv[j] = __shfl_sync(kFullMask, f0, sample_lane[j]);
            const f2 K2 = f2_splat(median5(kv[0], kv[1], kv[2], kv[3], kv[4]));
            f2 d[VPL][H];
            f2 as[2] = {f2_splat(0.f), f2_splat(0.f)}, ad[2] = {f2_splat(0.f), f2_splat(0.f)};
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                PR::unpack(sp[v], d[v]);
                if (v * 32 + lane < nvec) {
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        as[h & 1] = f2_add(as[h & 1], d[v][h]);
                        d[v][h] = f2_sub(d[v][h], K2);
                        ad[h & 1] = f2_add(ad[h & 1], d[v][h]);
                    }
                }
            }
            const f2 as2 = f2_add(as[0], as[1]), ad2 = f2_add(ad[0], ad[1]);
            float S = f2_lo(as2) + f2_hi(as2);
            float md = (f2_lo(ad2) + f2_hi(ad2)) * inv_lane;
            const f2 ml2 = f2_splat(md);
            f2 q[2] = {f2_splat(0.f), f2_splat(0.f)};
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                if (v * 32 + lane < nvec) {
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const f2 t = f2_sub(d[v][h], ml2);
                        q[h & 1] = f2_fma(t, t, q[h & 1]);
                    }
                }
            }
            const f2 q2 = f2_add(q[0], q[1]);
            float M2 = f2_lo(q2) + f2_hi(q2);
            if (equal)  // the one reduction of the row
                chan_reduce_equal(16, n_lane, S, md, M2);
            else
                chan_reduce_any(n_lane, S, md, M2);
            const float rs = rsqrtf(rdiv.div(M2) + eps);
            if (lane == 0) {
                mean[row] = rdiv.div(S);
                rstd[row] = rs;
            }
            // out = gamma * ((s - K - mean_d) * rs) + beta
            const f2 rs2 = f2_splat(rs), md2 = f2_splat(md);
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const int vi = v * 32 + lane;
                if (vi < nvec) {
                    f2 o[H];
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = f2_fma(gp[v][h], f2_mul(f2_sub(d[v][h], md2), rs2), bp[v][h]);
                    st_stream(out + base + (size_t)vi * V, PR::pack(o));
                }
            }
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
template <typename T, int VPT, bool HAS_RES>
__global__ void __launch_bounds__(kFwdBlockMaxThreads, 1)
    fwd_block_kernel(const T* __restrict__ x, const T* __restrict__ res,
                     const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                     int rows, int cols, T* __restrict__ out, T* __restrict__ res_out,
                     float* __restrict__ mean, float* __restrict__ rstd, int stages,
                     unsigned* status, uint64_t wait_limit_ns) {
    using IO = Io<T>;
    constexpr int V = IO::kVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages];
    __shared__ float red[3][32];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nw = nthreads >> 5;
    const int nvec = cols / V;
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned nin = HAS_RES ? 2u : 1u;
    const unsigned slot_bytes = nin * row_bytes;
    const RowDivisor rdiv(cols);

    // Counts of values in a row (the same for every row): this thread's, and in lane w the
    // count of warp w, whose summary lane w takes in the cross-warp butterfly.  When every
    // thread holds VPT vectors (and the warp count is a power of two) the butterflies merge
    // equal halves.
    auto vecs_of = [&](int t) {
        int n = 0;
#pragma unroll
        for (int v = 0; v < VPT; ++v) n += v * nthreads + t < nvec ? 1 : 0;
        return n;
    };
    const float n_thr = (float)(vecs_of(tid) * V);
    const float inv_thr = n_thr > 0.f ? 1.0f / n_thr : 0.f;
    int nv_warp = 0;
    for (int j = 0; j < 32 && lane < nw; ++j) nv_warp += vecs_of(lane * 32 + j);
    const float n_warp = (float)(nv_warp * V);
    const bool equal_thr = nvec == nthreads * VPT;
    const bool equal_warps = equal_thr && (nw & (nw - 1)) == 0;
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

    // gamma, beta for this thread's vectors (the same columns in every row), as fp32 pairs.
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 gp[VPT][H], bp[VPT][H];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int vi = v * nthreads + tid;
        PR::unpack(vi < nvec ? ld_keep(gamma + (size_t)vi * V) : make_uint4(0, 0, 0, 0), gp[v]);
        PR::unpack(vi < nvec ? ld_keep(beta + (size_t)vi * V) : make_uint4(0, 0, 0, 0), bp[v]);
    }

    const bool write_res = res_out != nullptr;
    int k = 0;
    RingPos pos;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, ++k, pos.next(stages)) {
        const int slot = pos.slot;
        if (!mbar_wait(&full_bar[slot], pos.phase, wait_limit_ns)) abort_flag = 1;
        const T* xs = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes);
        const T* rsm = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes + row_bytes);
        const size_t base = (size_t)row * cols;
        // The row's shift K: the median of five of its values, which every thread reads from
        // shared memory (first, so that these loads overlap the vector loads below).
        const f2 K2 = f2_splat(row_shift<T, HAS_RES>(xs, rsm, cols));

        uint4 sp[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)vi * V);
                sp[v] = HAS_RES ? IO::add_round(xv, *reinterpret_cast<const uint4*>(rsm + (size_t)vi * V))
                                : xv;
                if (write_res) st_stream(res_out + base + (size_t)vi * V, sp[v]);
            } else {
                sp[v] = make_uint4(0, 0, 0, 0);
            }
        }
        // This thread's summary: the plain sum of s, then d = s - K, the mean of d and M2
        // about it.  The low halves of the pairs take the even columns, the high halves the
        // odd ones.
        f2 d[VPT][H];
        f2 as = f2_splat(0.f), ad = f2_splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            PR::unpack(sp[v], d[v]);
            if (v * nthreads + tid < nvec) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    as = f2_add(as, d[v][h]);
                    d[v][h] = f2_sub(d[v][h], K2);
                    ad = f2_add(ad, d[v][h]);
                }
            }
        }
        float S = f2_lo(as) + f2_hi(as);
        float md = (f2_lo(ad) + f2_hi(ad)) * inv_thr;
        const f2 ml2 = f2_splat(md);
        f2 q = f2_splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            if (v * nthreads + tid < nvec) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const f2 t = f2_sub(d[v][h], ml2);
                    q = f2_fma(t, t, q);
                }
            }
        }
        float M2 = f2_lo(q) + f2_hi(q);
        if (equal_thr)
            chan_reduce_equal(16, n_thr, S, md, M2);
        else
            chan_reduce_any(n_thr, S, md, M2);
        if (lane == 0) {
            red[0][warp] = S;
            red[1][warp] = md;
            red[2][warp] = M2;
        }
        __syncthreads();  // the one cross-warp exchange of the row
        if (abort_flag) break;
        // Every warp merges the warps' summaries the same way: the same bits everywhere.
        if (equal_warps) {  // lane l takes warp l mod nw; groups of nw lanes merge alike
            const int w = lane & (nw - 1);
            S = red[0][w];
            md = red[1][w];
            M2 = red[2][w];
            chan_reduce_equal(nw >> 1, 32.f * n_thr, S, md, M2);
        } else {
            S = lane < nw ? red[0][lane] : 0.f;
            md = lane < nw ? red[1][lane] : 0.f;
            M2 = lane < nw ? red[2][lane] : 0.f;
            chan_reduce_any(n_warp, S, md, M2);
        }
        const float rs = rsqrtf(rdiv.div(M2) + eps);
        if (tid == 0) {
            mean[row] = rdiv.div(S);
            rstd[row] = rs;
        }
        // out = gamma * ((s - K - mean_d) * rs) + beta
        const f2 rs2 = f2_splat(rs), md2 = f2_splat(md);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int vi = v * nthreads + tid;
            if (vi < nvec) {
                f2 o[H];
#pragma unroll
                for (int h = 0; h < H; ++h)
                    o[h] = f2_fma(gp[v][h], f2_mul(f2_sub(d[v][h], md2), rs2), bp[v][h]);
                st_stream(out + base + (size_t)vi * V, PR::pack(o));
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
// second one hits L1/L2); the statistics are the same mergeable summaries.
// ---------------------------------------------------------------------------------------
template <typename T, bool HAS_RES>
__global__ void __launch_bounds__(kFwdScalarThreads)
    fwd_scalar_kernel(const T* __restrict__ x, const T* __restrict__ res,
                      const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                      int rows, int cols, T* __restrict__ out, T* __restrict__ res_out,
                      float* __restrict__ mean, float* __restrict__ rstd) {
    using IO = Io<T>;
    pdl_enter();
    constexpr int NW = kFwdScalarThreads / 32;
    __shared__ float red[3][NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const RowDivisor rdiv(cols);
    const bool write_res = res_out != nullptr;
    // This thread's count of values in a row (columns tid, tid + 256, ...) and the weights of
    // the warp's and of the cross-warp butterflies; every warp's count follows from cols.
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
        auto load_s = [&](int j) -> float {
            float v = IO::to_f(x[base + j]);
            if (HAS_RES) v = IO::round(v + IO::to_f(res[base + j]));
            return v;
        };
        const float K = row_shift<T, HAS_RES>(x + base, HAS_RES ? res + base : nullptr, cols);
        // This thread's summary of its values: their plain sum S, and Welford's running mean
        // and M2 of d = s - K.
        float S = 0.f, md = 0.f, M2 = 0.f, n = 0.f;
        for (int j = tid; j < cols; j += kFwdScalarThreads) {
            const float sv = load_s(j);
            if (write_res) res_out[base + j] = IO::from_f(sv);
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
            out[base + j] = IO::from_f(IO::to_f(gamma[j]) * ((sv - K - md) * rs) + IO::to_f(beta[j]));
        }
        __syncthreads();  // `red` is reused by the next row
    }
}

// ---------------------------------------------------------------------------------------
// Host-side dispatch.
// ---------------------------------------------------------------------------------------
template <typename T>
cudaError_t launch_warp(const FwdArgs& a, int vpl, cudaStream_t stream) {
    const void* kern = nullptr;
    const bool has_res = a.res != nullptr;
#define LNK_FWD_TILE_CASE(N)                                                               \
    case N:                                                                                \
        kern = has_res ? (const void*)fwd_tile_kernel<T, N, true>                          \
                       : (const void*)fwd_tile_kernel<T, N, false>;                        \
        break;
    switch (vpl) {
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
    const size_t slot_bytes = (size_t)(has_res ? 2 : 1) * kTileRows * a.cols * sizeof(T);
    // Two to four tiles in flight per block, two blocks per SM when they fit.
    int stages = (int)std::min<size_t>(kMaxStages, ((size_t)di.smem_optin / 2) / slot_bytes);
    stages = std::max(2, stages);
    const size_t smem = (size_t)stages * slot_bytes;
    if (smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int ntiles = (a.rows + kTileRows - 1) / kTileRows;
    const int occ = std::max(1, blocks_per_sm(kern, kTileThreads, smem));
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
    void* args[] = {&x,   &res,     &gamma, &beta, &eps,    &rows,   &cols,
                    &out, &res_out, &mean,  &rstd, &stages, &status, &limit};
    return launch_kernel(kern, dim3(grid), dim3(kTileThreads), smem, stream, args, false);
}

template <typename T>
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
        kern = has_res ? (const void*)fwd_block_kernel<T, N, true>                         \
                       : (const void*)fwd_block_kernel<T, N, false>;                       \
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
    void* args[] = {&x,   &res,     &gamma, &beta, &eps,   &rows,   &cols,
                    &out, &res_out, &mean,  &rstd, &stages, &status, &limit};
    return launch_kernel(kern, dim3(grid), dim3(threads), smem, stream, args, false);
}

template <typename T>
cudaError_t launch_scalar(const FwdArgs& a, cudaStream_t stream) {
    const bool has_res = a.res != nullptr;
    const void* kern = has_res ? (const void*)fwd_scalar_kernel<T, true>
                               : (const void*)fwd_scalar_kernel<T, false>;
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
    void* args[] = {&x, &res, &gamma, &beta, &eps, &rows, &cols, &out, &res_out, &mean, &rstd};
    return launch_kernel(kern, dim3(grid), dim3(kFwdScalarThreads), 0, stream, args, false);
}

template <typename T>
cudaError_t launch_fwd_t(const FwdArgs& a, bool aligned, int path, cudaStream_t stream) {
    constexpr int V = Io<T>::kVec;
    if (!aligned || path == kPathScalar) return launch_scalar<T>(a, stream);
    const int nvec = a.cols / V;
    const int vpl = (nvec + 31) / 32;
    if (path == kPathBlock) return launch_block<T>(a, stream);
    if (vpl <= 8) return launch_warp<T>(a, vpl, stream);
    return launch_block<T>(a, stream);
}

}  // namespace

cudaError_t launch_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                       cudaStream_t stream, int* launches) {
    *launches = 0;
    if (a.rows == 0) return cudaSuccess;
    cudaError_t e = dt == Dtype::F32 ? launch_fwd_t<float>(a, aligned, path_override, stream)
                                     : launch_fwd_t<__nv_bfloat16>(a, aligned, path_override, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
