// dropout.cu -- backward of the bias + dropout + residual prologue of the LayerNorm forward.
//
// The forward ("Accelerating Transformer on GPU (I)", section 2.3, fused into the LayerNorm
// forward kernels) computes s = res + keep * (h + bias) / (1 - p) with keep regenerated from
// a counter-based generator (Philox-4x32-10, see DropoutRng), so the backward can regenerate
// it, or read the bits the forward stored while it decided (1 bit per element, rows padded
// to whole bytes; "... (II)", section 3.2: the dropout backward needs the mask -- LightSeq
// keeps one byte per element).  Given ds, the gradient with respect to s (the LayerNorm backward's dx, which is also
// the residual's gradient):
//   dh = ds * keep / (1 - p),   dbias = sum over rows of dh.
// One cooperative launch.  A grid of (column tile) x (row segment) blocks of 256 threads
// (32 column slots x 8 row groups), one wave of resident blocks: a thread owns one 16-byte
// vector of columns (or one column, for rows that are not 16-byte multiples) and every 8th
// row of its segment, loads a batch of rows before it uses any (many bytes in flight per
// SM), writes dh and keeps Kahan-compensated column sums; the block folds its 8 row groups in
// order through shared memory and stores one (hi, lo) partial row slice per segment, as
// partials that announce themselves (ln_finish.cuh).  Then the first `segments` blocks each
// finish a slice of the columns: they read every segment's partials of their slice as they
// land and add them in segment order (TwoSum), zeroing what they read, so the workspace is
// left all zero.  The order of every addition depends only on (rows, cols, device), so dbias
// is bitwise reproducible; no float atomics, no second launch.
#include <algorithm>

#include "ln_device.cuh"
#include "ln_finish.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

constexpr int kDbX = 32, kDbY = 8;  // a block: column slots x row groups
constexpr int kDbThreads = kDbX * kDbY;
constexpr int kDbBatch = 4;         // rows a thread loads before it uses any
constexpr int kDbBlocksPerSm = 3;   // resident blocks (the registers allow 3)

// The finish (finish_units) reads its arguments by these names: one statistic, dbias as
// "dgamma".
struct DbParams {
    const void* ds;
    void* dh;
    void* dgamma;  // dbias
    void* dbeta;   // unused (one statistic)
    float2* part;  // [segments][cols] (hi, lo), announcing themselves
    int rows, cols, segs, ctiles;
    int nstat;     // 1
    int fin_rw;
    unsigned* status;
    uint64_t limit_ns;
    float scale;
    DropoutRng rng;
    const uint8_t* keep;  // the forward's stored keep bits (rows padded to bytes), or null
    int keep_stride;      // bytes per row of keep: ceil(cols / 8)
};

__device__ __forceinline__ void kahan_step(float& s, float& c, float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

// One 16-byte vector of ds (CV = Io<T>::kVec elements starting at element i0, i0 % CV == 0):
// dh = keep ? ds * scale : 0, stored, and added to the thread's column sums.
// The stored keep bits of the CV (4 or 8) columns from col0 of `row` (col0 % CV == 0): a
// byte, or half of one.
template <int CV, bool BITS>
__device__ __forceinline__ unsigned keep_bits_of(const DbParams& p, int row, int col0, size_t) {
    static_assert(BITS, "the generator's decisions are compared in drop_vec");
    const unsigned b = __ldg(p.keep + (size_t)row * p.keep_stride + (col0 >> 3));
    return CV == 8 ? b : (b >> (col0 & 4)) & 0xFu;
}

template <bool BITS>
__device__ __forceinline__ bool keep_one(const DbParams& p, int row, int col, size_t i) {
    if constexpr (BITS)
        return (__ldg(p.keep + (size_t)row * p.keep_stride + (col >> 3)) >> (col & 7)) & 1u;
    else
        return p.rng.keep(i);
}

template <typename T, int CV, bool BITS>
__device__ __forceinline__ uint4 drop_vec(const DbParams& p, const uint4& u, int row, int col0,
                                          size_t i0, float (&S)[CV], float (&C)[CV]) {
    using IO = Io<T>;
    float v[CV];
    IO::unpack(u, v);
    if constexpr (BITS) {
        const unsigned kb = keep_bits_of<CV, true>(p, row, col0, i0);
#pragma unroll
        for (int k = 0; k < CV; ++k) {
            v[k] = (kb >> k) & 1u ? __fmul_rn(v[k], p.scale) : 0.f;
            kahan_step(S[k], C[k], v[k]);
        }
    } else {  // the generator's words compared directly
        uint32_t w[CV];
        const uint4 wa = p.rng.words(i0 >> 2);
        w[0] = wa.x; w[1] = wa.y; w[2] = wa.z; w[3] = wa.w;
        if constexpr (CV == 8) {
            const uint4 wb = p.rng.words((i0 >> 2) + 1);
            w[4] = wb.x; w[5] = wb.y; w[6] = wb.z; w[7] = wb.w;
        }
#pragma unroll
        for (int k = 0; k < CV; ++k) {
            v[k] = w[k] >= p.rng.thr ? __fmul_rn(v[k], p.scale) : 0.f;
            kahan_step(S[k], C[k], v[k]);
        }
    }
    return IO::pack(v);
}

// CV = Io<T>::kVec adjacent columns per thread with 16-byte accesses (cols % CV == 0 and
// 16-byte aligned rows), or CV = 1 for any layout.  Column tiles are taken grid-stride, so
// the widest rows still fit in one resident wave.
template <typename T, int CV, bool BITS>
__global__ void __launch_bounds__(kDbThreads, kDbBlocksPerSm) dropout_bwd_kernel(const DbParams p) {
    using IO = Io<T>;
    __shared__ float2 fold[kDbY][kDbX * CV];
    __shared__ float scratch[kDbThreads * 4];  // the finish: 2 U floats per thread, U <= 2
    pdl_enter();
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int seg = blockIdx.y;
    const int r0 = (int)((long long)p.rows * seg / p.segs);
    const int r1 = (int)((long long)p.rows * (seg + 1) / p.segs);
    const T* ds = static_cast<const T*>(p.ds);
    T* dh = static_cast<T*>(p.dh);
    for (int ct = blockIdx.x; ct < p.ctiles; ct += gridDim.x) {  // block-uniform
        const int col0 = (ct * kDbX + tx) * CV;
        float S[CV], C[CV];
#pragma unroll
        for (int k = 0; k < CV; ++k) S[k] = C[k] = 0.f;
        if (col0 < p.cols) {
            int r = r0 + ty;
            if constexpr (CV > 1) {
                for (; r + (kDbBatch - 1) * kDbY < r1; r += kDbBatch * kDbY) {
                    uint4 u[kDbBatch];
#pragma unroll
                    for (int b = 0; b < kDbBatch; ++b)
                        u[b] = __ldcs(reinterpret_cast<const uint4*>(ds + (size_t)(r + b * kDbY) * p.cols + col0));
#pragma unroll
                    for (int b = 0; b < kDbBatch; ++b) {
                        const size_t i0 = (size_t)(r + b * kDbY) * p.cols + col0;
                        *reinterpret_cast<uint4*>(dh + i0) = drop_vec<T, CV, BITS>(p, u[b], r + b * kDbY, col0, i0, S, C);
                    }
                }
                for (; r < r1; r += kDbY) {
                    const size_t i0 = (size_t)r * p.cols + col0;
                    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(ds + i0));
                    *reinterpret_cast<uint4*>(dh + i0) = drop_vec<T, CV, BITS>(p, u, r, col0, i0, S, C);
                }
            } else {
                for (; r + (kDbBatch - 1) * kDbY < r1; r += kDbBatch * kDbY) {
                    float v[kDbBatch];
#pragma unroll
                    for (int b = 0; b < kDbBatch; ++b) v[b] = IO::to_f(ds[(size_t)(r + b * kDbY) * p.cols + col0]);
#pragma unroll
                    for (int b = 0; b < kDbBatch; ++b) {
                        const size_t i0 = (size_t)(r + b * kDbY) * p.cols + col0;
                        const float w = keep_one<BITS>(p, r + b * kDbY, col0, i0) ? __fmul_rn(v[b], p.scale) : 0.f;
                        dh[i0] = IO::from_f(w);
                        kahan_step(S[0], C[0], w);
                    }
                }
                for (; r < r1; r += kDbY) {
                    const size_t i0 = (size_t)r * p.cols + col0;
                    const float w = keep_one<BITS>(p, r, col0, i0) ? __fmul_rn(IO::to_f(ds[i0]), p.scale) : 0.f;
                    dh[i0] = IO::from_f(w);
                    kahan_step(S[0], C[0], w);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < CV; ++k) fold[ty][tx * CV + k] = make_float2(S[k], -C[k]);  // value S - C
        __syncthreads();
        // The 8 row groups' sums of each column, in row-group order: thread t folds column
        // slot t (and t + 256, ... for wider tiles), so the slice is stored with consecutive
        // addresses.
        for (int t = tid; t < kDbX * CV; t += kDbThreads) {
            const int c = ct * kDbX * CV + t;
            if (c >= p.cols) continue;
            float hs = 0.f, ls = 0.f;
#pragma unroll
            for (int g = 0; g < kDbY; ++g) comp_add(hs, ls, fold[g][t].x, fold[g][t].y);
            st_part2(p.part + (size_t)seg * p.cols + c, hs, ls);
        }
        __syncthreads();  // fold is reused by the next column tile
    }
    // The finish: the first `segs` blocks each own a slice of the column groups.
    const int f = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    if (f < p.segs) {
        if (p.cols % 2 == 0)
            finish_units<T, 2, false>(p, p.segs, p.segs, f, scratch);
        else
            finish_units<T, 1, false>(p, p.segs, p.segs, f, scratch);
    }
}

template <typename T>
cudaError_t launch_db_t(DbParams p, bool vec, cudaStream_t stream) {
    constexpr int kVec = Io<T>::kVec;
    const void* k1 = p.keep ? (vec ? (const void*)dropout_bwd_kernel<T, kVec, true>
                                   : (const void*)dropout_bwd_kernel<T, 1, true>)
                            : (vec ? (const void*)dropout_bwd_kernel<T, kVec, false>
                                   : (const void*)dropout_bwd_kernel<T, 1, false>);
    const int occ = std::max(1, blocks_per_sm(k1, kDbThreads, 0));
    const int slots = occ * device_info(-1).sms;  // blocks that can be resident at once
    const int gx = std::max(1, std::min(p.ctiles, slots / p.segs));
    if (gx * p.segs > slots) return cudaErrorCooperativeLaunchTooLarge;
    p.fin_rw = fin_warps_per_group(kDbThreads / 32, p.segs, 2 * (p.cols % 2 == 0 ? 2 : 1));
    void* args[] = {&p};
    // Cooperative: every block resident, as the finish's polls need.
    return launch_kernel(k1, dim3(gx, p.segs), dim3(kDbThreads), 0, stream, args, true);
}

}  // namespace

bool dropout_bwd_vector(Dtype dt, int cols, bool aligned) {
    return aligned && cols % (dt == Dtype::F32 ? 4 : 8) == 0;
}

// Segments of rows (partial rows of dbias): one wave of resident blocks over the column
// tiles, at least one batch of rows per row group (32 rows), and at most min(rows,
// kDbBlocksPerSm per SM) -- within the workspace bound of 8 per SM, and so that every
// segment has a resident block for at least one column tile.
int dropout_bwd_segments(int rows, int cols, int sms, int cv) {
    const int ctiles = (cols + kDbX * cv - 1) / (kDbX * cv);
    int segs = std::max(1, kDbBlocksPerSm * sms / ctiles);
    segs = std::min(segs, std::max(1, rows / (kDbY * kDbBatch)));
    return std::max(1, std::min(segs, std::min(rows, kDbBlocksPerSm * sms)));
}

cudaError_t launch_dropout_bwd(Dtype dt, const DropoutBwdArgs& a, bool vec, cudaStream_t stream,
                               int* launches) {
    *launches = 0;
    const int cv = vec ? (dt == Dtype::F32 ? 4 : 8) : 1;
    DbParams p;
    p.ds = a.ds;
    p.dh = a.dh;
    p.dgamma = a.dbias;
    p.dbeta = nullptr;
    p.part = reinterpret_cast<float2*>(a.partials);
    p.rows = a.rows;
    p.cols = a.cols;
    p.segs = a.segs;
    p.ctiles = (a.cols + kDbX * cv - 1) / (kDbX * cv);
    p.nstat = 1;
    p.fin_rw = 1;
    p.status = a.status;
    p.limit_ns = a.wait_limit_ns;
    p.scale = a.scale;
    p.rng = DropoutRng::make(a.seed, a.offset, a.thr);
    p.keep = a.keep;
    p.keep_stride = (a.cols + 7) / 8;
    cudaError_t e = dt == Dtype::F32 ? launch_db_t<float>(p, vec, stream)
                                     : launch_db_t<__nv_bfloat16>(p, vec, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
