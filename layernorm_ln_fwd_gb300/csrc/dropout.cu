// dropout.cu -- backward of the bias + dropout + residual prologue of the LayerNorm forward.
//
// The forward ("Accelerating Transformer on GPU (I)", section 2.3, fused into the LayerNorm
// forward kernels) computes s = res + keep * (h + bias) / (1 - p) with keep regenerated from
// a counter-based generator (Philox-4x32-10, see DropoutRng), so the backward needs no stored
// mask.  Given ds, the gradient with respect to s (the LayerNorm backward's dx, which is also
// the residual's gradient):
//   dh = ds * keep / (1 - p),   dbias = sum over rows of dh.
// dbias is reduced deterministically, without float atomics, in two launches: a grid of
// (column tile) x (row segment) blocks -- 32 x 8 threads, each thread CV adjacent columns and
// every 8th row of its segment, Kahan-compensated -- writes one (hi, lo) partial row per
// segment after folding its 8 row groups in order through shared memory; then one thread per
// column adds the segments' partials in segment order (TwoSum) and zeroes them, leaving the
// workspace all zero for the next call.  The order of every addition depends only on (rows,
// cols, device), so dbias is bitwise reproducible.
#include <algorithm>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

constexpr int kDbX = 32, kDbY = 8;

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

// CV = 4 adjacent columns per thread with vector loads (cols % 4 == 0, 16-byte aligned for
// fp32 / 8-byte for bf16), or CV = 1 for any layout.
template <typename T, int CV>
__global__ void __launch_bounds__(kDbX * kDbY) dropout_bwd_kernel(const DbParams p) {
    using IO = Io<T>;
    __shared__ float2 fold[kDbY][kDbX * CV];
    pdl_enter();
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int col0 = (blockIdx.x * kDbX + tx) * CV;
    const int seg = blockIdx.y;
    const int r0 = (int)((long long)p.rows * seg / p.segs), r1 = (int)((long long)p.rows * (seg + 1) / p.segs);
    const T* ds = static_cast<const T*>(p.ds);
    T* dh = static_cast<T*>(p.dh);
    float S[CV], C[CV];
#pragma unroll
    for (int k = 0; k < CV; ++k) S[k] = C[k] = 0.f;
    if (col0 < p.cols) {
        for (int r = r0 + ty; r < r1; r += kDbY) {
            const size_t i0 = (size_t)r * p.cols + col0;
            if constexpr (CV == 4) {
                float v[4];
                if constexpr (sizeof(T) == 4) {
                    const float4 u = *reinterpret_cast<const float4*>(ds + i0);
                    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
                } else {
                    const uint2 u = *reinterpret_cast<const uint2*>(ds + i0);
                    const float2 a = IO::pair(u.x), b = IO::pair(u.y);
                    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
                }
                const unsigned keep = p.rng.keep4(i0 >> 2);
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = ((keep >> k) & 1u) ? v[k] * p.scale : 0.f;
                if constexpr (sizeof(T) == 4) {
                    *reinterpret_cast<float4*>(dh + i0) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
                    *reinterpret_cast<uint2*>(dh + i0) = make_uint2(IO::pair_bits(v[0], v[1]), IO::pair_bits(v[2], v[3]));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) kahan_step(S[k], C[k], v[k]);
            } else {
                float v = IO::to_f(ds[i0]);
                v = p.rng.keep(i0) ? v * p.scale : 0.f;
                dh[i0] = IO::from_f(v);
                kahan_step(S[0], C[0], v);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < CV; ++k) fold[ty][tx * CV + k] = make_float2(S[k], -C[k]);  // value S - C
    __syncthreads();
    if (ty == 0 && col0 < p.cols) {
#pragma unroll
        for (int k = 0; k < CV; ++k) {
            float hs = 0.f, ls = 0.f;
            for (int g = 0; g < kDbY; ++g) two_sum_add(hs, ls, fold[g][tx * CV + k].x, fold[g][tx * CV + k].y);
            if (col0 + k < p.cols) p.part[(size_t)seg * p.cols + col0 + k] = make_float2(hs, ls);
        }
    }
}

template <typename T>
__global__ void dropout_bias_finish(const DbParams p) {
    using IO = Io<T>;
    pdl_enter();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= p.cols) return;
    float hs = 0.f, ls = 0.f;
    for (int g = 0; g < p.segs; ++g) {
        float2* q = p.part + (size_t)g * p.cols + c;
        const float2 v = *q;
        two_sum_add(hs, ls, v.x, v.y);
        *q = make_float2(0.f, 0.f);  // the workspace is left zero
    }
    static_cast<T*>(p.dbias)[c] = IO::from_f(hs + ls);
}

template <typename T>
cudaError_t launch_db_t(DbParams p, bool vec, cudaStream_t stream) {
    const int cv = vec ? 4 : 1;
    const int ctiles = (p.cols + kDbX * cv - 1) / (kDbX * cv);
    void* args[] = {&p};
    const void* k1 = vec ? (const void*)dropout_bwd_kernel<T, 4> : (const void*)dropout_bwd_kernel<T, 1>;
    cudaError_t e = launch_kernel(k1, dim3(ctiles, p.segs), dim3(kDbX, kDbY), 0, stream, args, false);
    if (e != cudaSuccess) return e;
    return launch_kernel((const void*)dropout_bias_finish<T>, dim3((p.cols + 255) / 256), dim3(256),
                         0, stream, args, false);
}

}  // namespace

// Segments of rows for the dbias partials: about two blocks per SM over the column tiles,
// at least 8 rows each, at most 8 per SM (the workspace bound).
int dropout_bwd_segments(int rows, int cols, int sms) {
    const int ctiles = (cols + kDbX - 1) / kDbX;  // an upper bound on the tiles of either form
    int segs = std::max(1, (2 * sms + ctiles - 1) / ctiles);
    segs = std::min(segs, std::max(1, rows / kDbY));
    return std::max(1, std::min(segs, 8 * sms));
}

cudaError_t launch_dropout_bwd(Dtype dt, const DropoutBwdArgs& a, bool aligned,
                               cudaStream_t stream, int* launches) {
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
    p.rng = DropoutRng{a.seed, a.offset, a.thr};
    const bool vec = aligned && a.cols % 4 == 0;
    cudaError_t e = dt == Dtype::F32 ? launch_db_t<float>(p, vec, stream)
                                     : launch_db_t<__nv_bfloat16>(p, vec, stream);
    if (e == cudaSuccess) *launches = 2;
    return e;
}

}  // namespace lnk
