// softmax.cu -- fused row softmax, forward and backward.
//
// Forward ("Accelerating Transformer on GPU (I)", section 4.1: scale, add the mask, row max,
// exponentiate, row sum, divide, all in one kernel):
//   z = scale * x + mask[r % mask_rows],  y = exp(z - max z) / sum exp(z - max z).
// The row is read once into registers.  A warp per row takes the page's two reductions (the
// row maximum, then the sum of exp(z - max)): one shuffle and one max or add per butterfly
// level.  A block per row merges its warps' (max, sum) pairs in ONE exchange through shared
// memory with the "online" merge m = max(ma, mb), s = sa exp(ma - m) + sb exp(mb - m), which
// saves a block barrier there.  The kernels work in base 2 -- z' = z log2(e) =
// (scale log2 e) x + mask log2 e, and exp(z - m) = exp2(z' - m') -- so that every
// exponential is one approximate base-2 exponent of the special-function unit (ex2_fast).
// Backward ("Accelerating Transformer on GPU (II)", section 3.1: only y is needed, one row
// reduction): dx = scale * y * (dy - sum dy y).
//
// Kernel families, as for the LayerNorm: warp per row fed by a bulk-copy (TMA) tile ring for
// rows of at most 256 vectors of 16 bytes (the page's lengths up to 2048 in bf16); a block
// per row, registers loaded with 128-bit loads, for longer rows; a scalar kernel for rows
// that are not 16-byte multiples or unaligned pointers.  Reductions are symmetric in their
// operands (max, commutative sums of separately rounded terms), so every lane ends with the
// same bits.  A row whose entries are all -inf gives NaN, as the definition does.
#include <algorithm>
#include <math.h>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

constexpr int kSmTileRows = 7;
constexpr int kSmTileThreads = (kSmTileRows + 1) * 32;
constexpr int kSmMaxStages = 4;
constexpr int kSmBlockThreads = 512;
constexpr int kSmScalarThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct SmParams {
    const void* a;       // x (forward) or dy (backward)
    const void* b;       // y (backward)
    const void* mask;    // forward: additive mask [mask_rows, cols], or null
    int mask_rows;
    float scale;
    int rows;
    int cols;
    void* out;           // y (forward) or dx (backward)
    int stages;
    unsigned* status;
    uint64_t limit_ns;
};

// The online merge of two (max, sum of exp(z - max)) pairs; a pair with max = -inf holds no
// finite value and sum 0.
__device__ __forceinline__ void online_merge(float& m, float& s, float mb, float sb) {
    const float mm = fmaxf(m, mb);
    if (mm == -INFINITY) {
        s = 0.f;
    } else {
        s = __fadd_rn(__fmul_rn(s, ex2_fast(m - mm)), __fmul_rn(sb, ex2_fast(mb - mm)));
    }
    m = mm;
}

__device__ __forceinline__ void warp_online(float& m, float& s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float mb = __shfl_xor_sync(kFullMask, m, o);
        const float sb = __shfl_xor_sync(kFullMask, s, o);
        online_merge(m, s, mb, sb);
    }
}

__device__ __forceinline__ float warp_sum1f(float a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(kFullMask, a, o);
    return a;
}

__device__ __forceinline__ float warp_max1f(float a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFullMask, a, o));
    return a;
}

// The forward of one row held by one warp, in the pages' two reductions ("Accelerating
// Transformer on GPU (I)", section 4.1): the row maximum M (one butterfly), then
// S = sum exp(z - M) (another), y = exp(z - M) / S.  Each butterfly level is one shuffle and
// one max or add -- against two exponentials and a rescale per level for the online merge --
// and the warp-per-row kernel runs enough warps per SM that instructions, not the second
// butterfly's latency, set its time.  Every lane ends with the same M and S (each level
// combines a pair commutatively).  A row whose entries are all -inf gives NaN (0 / 0).
template <typename T, int VPL, typename XS, typename MS, typename VALID, typename STORE>
__device__ __forceinline__ void warp_softmax_row(XS xs, MS ms, VALID valid, float scale,
                                                 STORE store) {
    using PR = Pairs<T>;
    constexpr int H = PR::kPairs;
    f2 z[VPL][H];
    float m = -INFINITY;
    const f2 a2 = f2_splat(scale * kLog2e), l2 = f2_splat(kLog2e);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        if (!valid(v)) continue;
        f2 xv[H], mv[H];
        PR::unpack(xs(v), xv);
        PR::unpack(ms(v), mv);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            // z' = (scale log2 e) x + mask log2 e: the score in base 2.
            z[v][h] = f2_fma(a2, xv[h], f2_mul(mv[h], l2));
            m = fmaxf(m, fmaxf(f2_lo(z[v][h]), f2_hi(z[v][h])));
        }
    }
    const float M = warp_max1f(m);
    const f2 nM = f2_splat(M == -INFINITY ? 0.f : -M);
    f2 acc = f2_splat(0.f);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        if (!valid(v)) continue;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const f2 t = f2_add(z[v][h], nM);
            z[v][h] = f2_make(ex2_fast(f2_lo(t)), ex2_fast(f2_hi(t)));
            acc = f2_add(acc, z[v][h]);
        }
    }
    const float S = warp_sum1f(f2_lo(acc) + f2_hi(acc));
    const f2 c2 = f2_splat(M == -INFINITY ? __int_as_float(0x7fc00000) : 1.0f / S);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        if (!valid(v)) continue;
        f2 o[H];
#pragma unroll
        for (int h = 0; h < H; ++h) o[h] = f2_mul(z[v][h], c2);
        store(v, PR::pack(o));
    }
}

// The forward of one row held as VPL vectors per lane (lane l: vectors l, l + stride, ...):
// `xs(v)` gives vector v's raw x, `valid(v)` whether it exists, `store(v, y)` writes y.
// The reduction is over the lanes of the warp (`warp_only`) or, for a block per row, the
// caller merges the warps' pairs.
template <typename T, int VPL>
struct SmRow {
    static constexpr int H = Pairs<T>::kPairs;
    float e[VPL][2 * H];  // exp(z - m_lane)
    float m = -INFINITY, s = 0.f;

    template <typename XS, typename MS, typename VALID>
    __device__ __forceinline__ void local(XS xs, MS ms, VALID valid, float scale) {
        f2 z[VPL][H];
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            if (!valid(v)) continue;
            f2 xv[H], mv[H];
            Pairs<T>::unpack(xs(v), xv);
            Pairs<T>::unpack(ms(v), mv);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                // z' = (scale log2 e) x + mask log2 e: the score in base 2.
                z[v][h] = f2_fma(f2_splat(scale * kLog2e), xv[h], f2_mul(mv[h], f2_splat(kLog2e)));
                m = fmaxf(m, fmaxf(f2_lo(z[v][h]), f2_hi(z[v][h])));
            }
        }
        // A lane whose values are all -inf (masked) keeps e = 0 and s = 0.
        const float sh = m == -INFINITY ? 0.f : m;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            if (!valid(v)) continue;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                e[v][2 * h] = ex2_fast(f2_lo(z[v][h]) - sh);
                e[v][2 * h + 1] = ex2_fast(f2_hi(z[v][h]) - sh);
                acc0 += e[v][2 * h];
                acc1 += e[v][2 * h + 1];
            }
        }
        s = acc0 + acc1;
    }

    // y of vector v once the row's max M and sum S are known.
    __device__ __forceinline__ uint4 y(int v, float c) const {
        f2 o[H];
#pragma unroll
        for (int h = 0; h < H; ++h) o[h] = f2_mul(f2_make(e[v][2 * h], e[v][2 * h + 1]), f2_splat(c));
        return Pairs<T>::pack(o);
    }
};

// ---------------------------------------------------------------------------------------
// Warp per row, fed by a bulk-copy tile ring (the LayerNorm tile kernel's pipeline): a
// producer warp copies tiles of 7 consecutive rows of each input, consumer warp w handles
// row w of every tile.  BWD: inputs dy and y; forward: input x (its mask rows, small and
// shared by many rows, are read through the cache).
// ---------------------------------------------------------------------------------------
template <typename T, int VPL, bool BWD>
__global__ void __launch_bounds__(kSmTileThreads, VPL <= 4 ? 2 : 1) sm_tile_kernel(const SmParams p) {
    constexpr int V = Io<T>::kVec;
    constexpr int NIN = BWD ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[kSmMaxStages], empty_bar[kSmMaxStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = p.rows, cols = p.cols, stages = p.stages;
    const int nvec = cols / V;
    const unsigned row_bytes = (unsigned)cols * (unsigned)sizeof(T);
    const unsigned tile_bytes = (unsigned)kSmTileRows * row_bytes;
    const unsigned slot_bytes = NIN * tile_bytes;
    const int ntiles = (rows + kSmTileRows - 1) / kSmTileRows;
    const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const T* M = static_cast<const T*>(p.mask);
    T* out = static_cast<T*>(p.out);

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kSmTileRows);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter();

    if (warp == kSmTileRows) {  // producer
        if (lane == 0) {
            int k = 0;
            RingPos pos;
            for (; k < my_tiles; ++k, pos.next(stages)) {
                const int slot = pos.slot;
                if (k >= stages && !mbar_wait(&empty_bar[slot], pos.phase ^ 1u, p.limit_ns)) {
                    raise_status(p.status, kStatusTimeout);
                    break;
                }
                const int r0 = ((int)blockIdx.x + k * (int)gridDim.x) * kSmTileRows;
                const unsigned bytes = (unsigned)min(kSmTileRows, rows - r0) * row_bytes;
                unsigned char* dst = smem_raw + (size_t)slot * slot_bytes;
                mbar_arrive_expect_tx(&full_bar[slot], NIN * bytes);
                bulk_g2s(dst, A + (size_t)r0 * cols, bytes, &full_bar[slot]);
                if (BWD) bulk_g2s(dst + tile_bytes, B + (size_t)r0 * cols, bytes, &full_bar[slot]);
            }
            for (int j = max(0, k - stages); j < k; ++j)
                (void)mbar_wait(&full_bar[j % stages], (unsigned)(j / stages) & 1u, p.limit_ns);
        }
        return;
    }

    const RowDivisor rdiv(cols);
    (void)rdiv;
    // Forward: the mask vectors of this warp's row of step k + 1 are loaded during step k
    // (the mask is read through the cache, and its load latency would otherwise stall every
    // row after its tile has landed).
    uint4 mk[BWD ? 1 : VPL];
    auto load_mask = [&](int kk) {
        if constexpr (!BWD) {
            const int r = ((int)blockIdx.x + kk * (int)gridDim.x) * kSmTileRows + warp;
            const T* mrow = M && kk < my_tiles && r < rows ? M + (size_t)(r % p.mask_rows) * cols
                                                          : nullptr;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                mk[v] = mrow && v * 32 + lane < nvec ? ld_keep(mrow + (size_t)(v * 32 + lane) * V)
                                                     : make_uint4(0, 0, 0, 0);
        }
    };
    load_mask(0);
    RingPos pos;
    for (int k = 0; k < my_tiles; ++k, pos.next(stages)) {
        const int slot = pos.slot;
        uint4 mcur[BWD ? 1 : VPL];
        if constexpr (!BWD) {
#pragma unroll
            for (int v = 0; v < VPL; ++v) mcur[v] = mk[v];
            load_mask(k + 1);
        }
        const bool ok = mbar_wait(&full_bar[slot], pos.phase, p.limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            if (lane == 0) raise_status(p.status, kStatusTimeout);
            break;
        }
        const int row = ((int)blockIdx.x + k * (int)gridDim.x) * kSmTileRows + warp;
        if (row < rows) {
            const size_t base = (size_t)row * cols;
            const T* as = reinterpret_cast<const T*>(smem_raw + (size_t)slot * slot_bytes +
                                                     (size_t)warp * row_bytes);
            auto valid = [&](int v) { return v * 32 + lane < nvec; };
            auto vec = [&](const T* rowp, int v) {
                return *reinterpret_cast<const uint4*>(rowp + (size_t)(v * 32 + lane) * V);
            };
            if constexpr (BWD) {
                const T* ys = as + (size_t)kSmTileRows * cols;
                constexpr int H = Pairs<T>::kPairs;
                f2 acc = f2_splat(0.f);
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    if (!valid(v)) continue;
                    f2 d[H], yv[H];
                    Pairs<T>::unpack(vec(as, v), d);
                    Pairs<T>::unpack(vec(ys, v), yv);
#pragma unroll
                    for (int h = 0; h < H; ++h) acc = f2_fma(d[h], yv[h], acc);
                }
                const f2 s2 = f2_splat(warp_sum1f(f2_lo(acc) + f2_hi(acc)));  // one reduction
                const f2 sc2 = f2_splat(p.scale);
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    if (!valid(v)) continue;
                    f2 d[H], yv[H], o[H];
                    Pairs<T>::unpack(vec(as, v), d);
                    Pairs<T>::unpack(vec(ys, v), yv);
#pragma unroll
                    for (int h = 0; h < H; ++h) o[h] = f2_mul(sc2, f2_mul(yv[h], f2_sub(d[h], s2)));
                    st_stream(out + base + (size_t)(v * 32 + lane) * V, Pairs<T>::pack(o));
                }
            } else {
                warp_softmax_row<T, VPL>(
                    [&](int v) { return vec(as, v); }, [&](int v) { return mcur[v]; },
                    valid, p.scale,
                    [&](int v, const uint4& y) { st_stream(out + base + (size_t)(v * 32 + lane) * V, y); });
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
}

// ---------------------------------------------------------------------------------------
// Block per row (rows longer than a warp's 256 vectors): thread t holds vectors t, t + T, ...
// of the row in registers (128-bit loads straight from global memory); the warps' partial
// results meet once in shared memory, and every thread merges them in the same order.
// ---------------------------------------------------------------------------------------
template <typename T, int VPT, bool BWD>
__global__ void __launch_bounds__(kSmBlockThreads, 1) sm_block_kernel(const SmParams p) {
    constexpr int V = Io<T>::kVec;
    constexpr int H = Pairs<T>::kPairs;
    __shared__ float red[2][32];
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nw = nthreads >> 5;
    const int cols = p.cols, nvec = cols / V;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const T* M = static_cast<const T*>(p.mask);
    T* out = static_cast<T*>(p.out);
    auto valid = [&](int v) { return v * nthreads + tid < nvec; };
    auto at = [&](const T* rowp, int v) { return rowp + (size_t)(v * nthreads + tid) * V; };
    auto at_out = [&](size_t base, int v) { return out + base + (size_t)(v * nthreads + tid) * V; };
    for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const size_t base = (size_t)row * cols;
        if constexpr (BWD) {
            f2 d[VPT][H], yv[VPT][H];
            f2 acc = f2_splat(0.f);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (!valid(v)) continue;
                Pairs<T>::unpack(__ldcs(reinterpret_cast<const uint4*>(at(A + base, v))), d[v]);
                Pairs<T>::unpack(__ldcs(reinterpret_cast<const uint4*>(at(B + base, v))), yv[v]);
#pragma unroll
                for (int h = 0; h < H; ++h) acc = f2_fma(d[v][h], yv[v][h], acc);
            }
            float s = warp_sum1f(f2_lo(acc) + f2_hi(acc));
            if (lane == 0) red[0][warp] = s;
            __syncthreads();
            s = 0.f;
            for (int w = 0; w < nw; ++w) s += red[0][w];
            const f2 s2 = f2_splat(s), sc2 = f2_splat(p.scale);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (!valid(v)) continue;
                f2 o[H];
#pragma unroll
                for (int h = 0; h < H; ++h) o[h] = f2_mul(sc2, f2_mul(yv[v][h], f2_sub(d[v][h], s2)));
                st_stream(at_out(base, v), Pairs<T>::pack(o));
            }
        } else {
            const T* mrow = M ? M + (size_t)(row % p.mask_rows) * cols : nullptr;
            SmRow<T, VPT> r;
            r.local([&](int v) { return __ldcs(reinterpret_cast<const uint4*>(at(A + base, v))); },
                    [&](int v) { return mrow ? ld_keep(at(mrow, v)) : make_uint4(0, 0, 0, 0); },
                    valid, p.scale);
            float mw = r.m, sw = r.s;
            warp_online(mw, sw);
            if (lane == 0) {
                red[0][warp] = mw;
                red[1][warp] = sw;
            }
            __syncthreads();  // the one cross-warp exchange of the row
            float mb = red[0][0], sb = red[1][0];
            for (int w = 1; w < nw; ++w) online_merge(mb, sb, red[0][w], red[1][w]);
            const float c = mb == -INFINITY ? __int_as_float(0x7fc00000)
                                            : (r.m == -INFINITY ? 0.f : ex2_fast(r.m - mb) / sb);
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (valid(v)) st_stream(at_out(base, v), r.y(v, c));
        }
        __syncthreads();  // `red` is reused by the next row
    }
}

// ---------------------------------------------------------------------------------------
// Scalar block per row: any alignment, any width.  Forward in two passes over the row (the
// second one hits L1/L2): per-thread online (max, sum) pairs merged over the block, then
// y = exp(z - M) / S.
// ---------------------------------------------------------------------------------------
template <typename T, bool BWD>
__global__ void __launch_bounds__(kSmScalarThreads) sm_scalar_kernel(const SmParams p) {
    using IO = Io<T>;
    constexpr int NW = kSmScalarThreads / 32;
    __shared__ float red[2][NW];
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = p.cols;
    const T* A = static_cast<const T*>(p.a);
    const T* B = static_cast<const T*>(p.b);
    const T* M = static_cast<const T*>(p.mask);
    T* out = static_cast<T*>(p.out);
    for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const size_t base = (size_t)row * cols;
        if constexpr (BWD) {
            float s = 0.f;
            for (int j = tid; j < cols; j += kSmScalarThreads)
                s = __fmaf_rn(IO::to_f(A[base + j]), IO::to_f(B[base + j]), s);
            s = warp_sum1f(s);
            if (lane == 0) red[0][warp] = s;
            __syncthreads();
            s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += red[0][w];
            for (int j = tid; j < cols; j += kSmScalarThreads) {
                const float yv = IO::to_f(B[base + j]);
                out[base + j] = IO::from_f(p.scale * (yv * (IO::to_f(A[base + j]) - s)));
            }
        } else {
            const T* mrow = M ? M + (size_t)(row % p.mask_rows) * cols : nullptr;
            auto z = [&](int j) {  // in base 2
                return __fmaf_rn(p.scale * kLog2e, IO::to_f(A[base + j]),
                                 mrow ? IO::to_f(mrow[j]) * kLog2e : 0.f);
            };
            float m = -INFINITY, s = 0.f;
            for (int j = tid; j < cols; j += kSmScalarThreads) online_merge(m, s, z(j), 1.f);
            warp_online(m, s);
            if (lane == 0) {
                red[0][warp] = m;
                red[1][warp] = s;
            }
            __syncthreads();
            m = red[0][0];
            s = red[1][0];
            for (int w = 1; w < NW; ++w) online_merge(m, s, red[0][w], red[1][w]);
            const float inv = 1.0f / s;
            for (int j = tid; j < cols; j += kSmScalarThreads)
                out[base + j] = IO::from_f(m == -INFINITY ? __int_as_float(0x7fc00000)
                                                          : ex2_fast(z(j) - m) * inv);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------------
template <typename T, bool BWD>
const void* sm_tile_for(int vpl) {
    switch (vpl) {
        case 1: return (const void*)sm_tile_kernel<T, 1, BWD>;
        case 2: return (const void*)sm_tile_kernel<T, 2, BWD>;
        case 3: return (const void*)sm_tile_kernel<T, 3, BWD>;
        case 4: return (const void*)sm_tile_kernel<T, 4, BWD>;
        case 5: return (const void*)sm_tile_kernel<T, 5, BWD>;
        case 6: return (const void*)sm_tile_kernel<T, 6, BWD>;
        case 7: return (const void*)sm_tile_kernel<T, 7, BWD>;
        case 8: return (const void*)sm_tile_kernel<T, 8, BWD>;
        default: return nullptr;
    }
}

template <typename T, bool BWD>
const void* sm_block_for(int vpt) {
    if (Io<T>::kVec == 8 && vpt > 4) return nullptr;  // bf16 rows of <= 16384 need <= 4
    switch (vpt) {
        case 1: return (const void*)sm_block_kernel<T, 1, BWD>;
        case 2: return (const void*)sm_block_kernel<T, 2, BWD>;
        case 3: return (const void*)sm_block_kernel<T, 3, BWD>;
        case 4: return (const void*)sm_block_kernel<T, 4, BWD>;
        default: break;
    }
    if constexpr (Io<T>::kVec == 4) {
        switch (vpt) {
            case 5: return (const void*)sm_block_kernel<T, 5, BWD>;
            case 6: return (const void*)sm_block_kernel<T, 6, BWD>;
            case 7: return (const void*)sm_block_kernel<T, 7, BWD>;
            case 8: return (const void*)sm_block_kernel<T, 8, BWD>;
            default: break;
        }
    }
    return nullptr;
}

template <typename T, bool BWD>
cudaError_t launch_sm_t(SmParams p, bool aligned, int path, cudaStream_t stream) {
    constexpr int V = Io<T>::kVec;
    const DeviceInfo& di = device_info(-1);
    void* args[] = {&p};
    const int nvec = p.cols / V;
    const int vpl = (nvec + 31) / 32;
    if (aligned && path != kPathScalar && path != kPathBlock && vpl <= 8) {
        const void* kern = sm_tile_for<T, BWD>(vpl);
        const size_t slot = (size_t)(BWD ? 2 : 1) * kSmTileRows * p.cols * sizeof(T);
        int stages = (int)std::min<size_t>(kSmMaxStages, ((size_t)di.smem_optin / 2) / slot);
        stages = std::max(2, stages);
        const size_t smem = (size_t)stages * slot;
        if (smem > (size_t)di.smem_optin) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        p.stages = stages;
        const int ntiles = (p.rows + kSmTileRows - 1) / kSmTileRows;
        const int occ = std::max(1, blocks_per_sm(kern, kSmTileThreads, smem));
        const int grid = std::max(1, std::min(ntiles, di.sms * occ));
        return launch_kernel(kern, dim3(grid), dim3(kSmTileThreads), smem, stream, args, false);
    }
    if (aligned && path != kPathScalar) {
        // 512 threads at most; the fewest vectors per thread that fit (cols <= 16384).
        const int vpt = (nvec + kSmBlockThreads - 1) / kSmBlockThreads;
        const int threads = std::max(32, ((nvec + vpt - 1) / vpt + 31) / 32 * 32);
        const void* kern = sm_block_for<T, BWD>(vpt);
        if (!kern) return cudaErrorInvalidValue;
        const int occ = std::max(1, blocks_per_sm(kern, threads, 0));
        const int grid = std::max(1, std::min(p.rows, di.sms * occ));
        return launch_kernel(kern, dim3(grid), dim3(threads), 0, stream, args, false);
    }
    const void* kern = (const void*)sm_scalar_kernel<T, BWD>;
    const int occ = std::max(1, blocks_per_sm(kern, kSmScalarThreads, 0));
    const int grid = std::max(1, std::min(p.rows, di.sms * occ));
    return launch_kernel(kern, dim3(grid), dim3(kSmScalarThreads), 0, stream, args, false);
}

}  // namespace

cudaError_t launch_softmax(Dtype dt, bool bwd, const SoftmaxArgs& a, bool aligned,
                           int path_override, cudaStream_t stream, int* launches) {
    *launches = 0;
    if (a.rows == 0) return cudaSuccess;
    SmParams p;
    p.a = a.a;
    p.b = a.b;
    p.mask = a.mask;
    p.mask_rows = a.mask_rows > 0 ? a.mask_rows : 1;
    p.scale = a.scale;
    p.rows = a.rows;
    p.cols = a.cols;
    p.out = a.out;
    p.stages = 0;
    p.status = a.status;
    p.limit_ns = a.wait_limit_ns;
    cudaError_t e;
    if (dt == Dtype::F32)
        e = bwd ? launch_sm_t<float, true>(p, aligned, path_override, stream)
                : launch_sm_t<float, false>(p, aligned, path_override, stream);
    else
        e = bwd ? launch_sm_t<__nv_bfloat16, true>(p, aligned, path_override, stream)
                : launch_sm_t<__nv_bfloat16, false>(p, aligned, path_override, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
