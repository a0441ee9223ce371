// dropout.cu -- backward of the bias + dropout + residual prologue of the LayerNorm forward.
//
// The forward ("Accelerating Transformer on GPU (I)", section 2.3, fused into the LayerNorm
// forward kernels) computes s = res + keep * (h + bias) / (1 - p) with keep regenerated from
// a counter-based generator (Philox-4x32-10, see DropoutRng), so the backward needs no stored
// mask.  Given ds, the gradient with respect to s (the LayerNorm backward's dx, which is also
// the residual's gradient):
//   dh = ds * keep / (1 - p),   dbias = sum over rows of dh.
// dbias is reduced deterministically, without float atomics, in two launches.  The first is
// a grid of (column tile) x (row segment) blocks of 32 x 8 threads, one wave of three blocks
// per SM:
// a thread owns one 16-byte vector of columns (or one column, for rows that are not
// 16-byte multiples) and every 8th row of its segment, loads a batch of rows before it uses
// any (many bytes in flight per SM), writes dh and keeps Kahan-compensated column sums; the
// block folds its 8 row groups in order through shared memory and writes one (hi, lo)
// partial row per segment.  The second launch adds, for each column, the segments' partials:
// 16 threads per column each take every 16th segment with all their loads issued at once,
// then the 16 sums are folded in order (TwoSum throughout); every partial read is zeroed,
// leaving the workspace all zero for the next call.  The order of every addition depends
// only on (rows, cols, device), so dbias is bitwise reproducible.
#include <algorithm>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

constexpr int kDbX = 32, kDbY = 8;  // the first launch's block: columns x row groups
constexpr int kDbBatch = 4;         // rows a thread loads before it uses any
constexpr int kDbBlocksPerSm = 3;   // resident blocks of the first launch (its registers allow 3)
constexpr int kFinY = 16;           // the finish's threads per column
constexpr int kFinBatch = 8;        // partials a finish thread loads before it adds any

struct DbParams {
    const void* ds;
    void* dh;
    void* dbias;
    float2* part;  // [segments][cols] (hi, lo)
    int rows, cols, segs;
    float scale;
    DropoutRng rng;
};

__device__ __forceinline__ void kahan_step(float& s, float& c, float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

__device__ __forceinline__ void two_sum_add(float& S, float& C, float h, float l) {
    float s, e;
    two_sum_f(S, h, s, e);
    S = s;
    C = __fadd_rn(C, __fadd_rn(e, l));
}

// One 16-byte vector of ds (CV = Io<T>::kVec elements starting at element i0, i0 % CV == 0):
// dh = keep ? ds * scale : 0, stored, and added to the thread's column sums.
template <typename T, int CV>
__device__ __forceinline__ uint4 drop_vec(const DbParams& p, const uint4& u, size_t i0,
                                          float (&S)[CV], float (&C)[CV]) {
    using IO = Io<T>;
    float v[CV];
    IO::unpack(u, v);
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
    return IO::pack(v);
}

// CV = Io<T>::kVec adjacent columns per thread with 16-byte accesses (cols % CV == 0 and
// 16-byte aligned rows), or CV = 1 for any layout.
template <typename T, int CV>
__global__ void __launch_bounds__(kDbX * kDbY, kDbBlocksPerSm) dropout_bwd_kernel(const DbParams p) {
    using IO = Io<T>;
    __shared__ float2 fold[kDbY][kDbX * CV];
    pdl_enter();
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int col0 = (blockIdx.x * kDbX + tx) * CV;
    const int seg = blockIdx.y;
    const int r0 = (int)((long long)p.rows * seg / p.segs);
    const int r1 = (int)((long long)p.rows * (seg + 1) / p.segs);
    const T* ds = static_cast<const T*>(p.ds);
    T* dh = static_cast<T*>(p.dh);
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
                    *reinterpret_cast<uint4*>(dh + i0) = drop_vec<T, CV>(p, u[b], i0, S, C);
                }
            }
            for (; r < r1; r += kDbY) {
                const size_t i0 = (size_t)r * p.cols + col0;
                const uint4 u = __ldcs(reinterpret_cast<const uint4*>(ds + i0));
                *reinterpret_cast<uint4*>(dh + i0) = drop_vec<T, CV>(p, u, i0, S, C);
            }
        } else {
            for (; r + (kDbBatch - 1) * kDbY < r1; r += kDbBatch * kDbY) {
                float v[kDbBatch];
#pragma unroll
                for (int b = 0; b < kDbBatch; ++b) v[b] = IO::to_f(ds[(size_t)(r + b * kDbY) * p.cols + col0]);
#pragma unroll
                for (int b = 0; b < kDbBatch; ++b) {
                    const size_t i0 = (size_t)(r + b * kDbY) * p.cols + col0;
                    const float w = p.rng.keep(i0) ? __fmul_rn(v[b], p.scale) : 0.f;
                    dh[i0] = IO::from_f(w);
                    kahan_step(S[0], C[0], w);
                }
            }
            for (; r < r1; r += kDbY) {
                const size_t i0 = (size_t)r * p.cols + col0;
                const float w = p.rng.keep(i0) ? __fmul_rn(IO::to_f(ds[i0]), p.scale) : 0.f;
                dh[i0] = IO::from_f(w);
                kahan_step(S[0], C[0], w);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < CV; ++k) fold[ty][tx * CV + k] = make_float2(S[k], -C[k]);  // value S - C
    __syncthreads();
    // The 8 row groups' sums of each column, in row-group order: thread t of the block folds
    // column slot t (and t + 256, ... for wider tiles), so the partial row is written by all
    // threads with consecutive addresses.
    for (int t = ty * kDbX + tx; t < kDbX * CV; t += kDbX * kDbY) {
        const int c = blockIdx.x * kDbX * CV + t;
        if (c >= p.cols) continue;
        float hs = 0.f, ls = 0.f;
#pragma unroll
        for (int g = 0; g < kDbY; ++g) two_sum_add(hs, ls, fold[g][t].x, fold[g][t].y);
        p.part[(size_t)seg * p.cols + c] = make_float2(hs, ls);
    }
}

// Column c's dbias: thread (tx, ty) adds segments ty, ty + 16, ... (kFinBatch loads in
// flight at a time), the 16 sums are folded in ty order; every partial read is zeroed.
template <typename T>
__global__ void __launch_bounds__(kDbX * kFinY) dropout_bias_finish(const DbParams p) {
    using IO = Io<T>;
    __shared__ float2 fold[kFinY][kDbX];
    pdl_enter();
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int c = blockIdx.x * kDbX + tx;
    float hs = 0.f, ls = 0.f;
    if (c < p.cols) {
        for (int g0 = ty; g0 < p.segs; g0 += kFinY * kFinBatch) {
            float2 v[kFinBatch];
#pragma unroll
            for (int b = 0; b < kFinBatch; ++b) {
                const int g = g0 + b * kFinY;
                v[b] = g < p.segs ? p.part[(size_t)g * p.cols + c] : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < kFinBatch; ++b) {
                const int g = g0 + b * kFinY;
                if (g < p.segs) p.part[(size_t)g * p.cols + c] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < kFinBatch; ++b) two_sum_add(hs, ls, v[b].x, v[b].y);
        }
    }
    fold[ty][tx] = make_float2(hs, ls);
    __syncthreads();
    if (ty == 0 && c < p.cols) {
        float H = 0.f, L = 0.f;
#pragma unroll
        for (int g = 0; g < kFinY; ++g) two_sum_add(H, L, fold[g][tx].x, fold[g][tx].y);
        static_cast<T*>(p.dbias)[c] = IO::from_f(H + L);
    }
}

template <typename T>
cudaError_t launch_db_t(DbParams p, bool vec, cudaStream_t stream) {
    constexpr int kVec = Io<T>::kVec;
    const int cv = vec ? kVec : 1;
    const int ctiles = (p.cols + kDbX * cv - 1) / (kDbX * cv);
    void* args[] = {&p};
    const void* k1 = vec ? (const void*)dropout_bwd_kernel<T, kVec> : (const void*)dropout_bwd_kernel<T, 1>;
    cudaError_t e = launch_kernel(k1, dim3(ctiles, p.segs), dim3(kDbX, kDbY), 0, stream, args, false);
    if (e != cudaSuccess) return e;
    return launch_kernel((const void*)dropout_bias_finish<T>, dim3((p.cols + kDbX - 1) / kDbX),
                         dim3(kDbX, kFinY), 0, stream, args, false);
}

}  // namespace

bool dropout_bwd_vector(Dtype dt, int cols, bool aligned) {
    return aligned && cols % (dt == Dtype::F32 ? 4 : 8) == 0;
}

// Segments of rows for the dbias partials: one wave of resident blocks over the column
// tiles, at least one batch of rows per row group (32 rows), at most min(rows, 8 per SM)
// segments (the workspace bound).
int dropout_bwd_segments(int rows, int cols, int sms, int cv) {
    const int ctiles = (cols + kDbX * cv - 1) / (kDbX * cv);
    int segs = std::max(1, kDbBlocksPerSm * sms / ctiles);
    segs = std::min(segs, std::max(1, rows / (kDbY * kDbBatch)));
    return std::max(1, std::min(segs, std::min(rows, 8 * sms)));
}

cudaError_t launch_dropout_bwd(Dtype dt, const DropoutBwdArgs& a, bool vec, cudaStream_t stream,
                               int* launches) {
    *launches = 0;
    DbParams p;
    p.ds = a.ds;
    p.dh = a.dh;
    p.dbias = a.dbias;
    p.part = reinterpret_cast<float2*>(a.partials);
    p.rows = a.rows;
    p.cols = a.cols;
    p.segs = a.segs;
    p.scale = a.scale;
    p.rng = DropoutRng::make(a.seed, a.offset, a.thr);
    cudaError_t e = dt == Dtype::F32 ? launch_db_t<float>(p, vec, stream)
                                     : launch_db_t<__nv_bfloat16>(p, vec, stream);
    if (e == cudaSuccess) *launches = 2;
    return e;
}

}  // namespace lnk
