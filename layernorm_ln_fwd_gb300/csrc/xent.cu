// xent.cu -- fused cross-entropy with label smoothing, forward and backward in one kernel.
//
// Per row of V logits x with target t ("Accelerating Transformer on GPU (I)", section 5.2;
// the fused classifier of "llm.c: the llmc/ CUDA kernel layer", section 6):
//   p = (1 - alpha) onehot(t) + alpha / V,  q = softmax(x),
//   loss = log Z + m - [(1 - alpha) x_t + (alpha / V) sum x],  dx = dloss * (q - p),
// with m = max x, Z = sum exp(x - m).  A block owns a row at a time: pass 1 reads the row
// once from HBM and reduces the online pair (max, sum of exp(x - max)), the plain sum of x
// and x_t in one block reduction; pass 2 reads the row again (from L2: the rows in flight
// are a small part of it) and writes dx, which may overwrite the logits in place (every
// element is read in pass 2 by the thread that writes it, after the whole block has finished
// pass 1).  exp(x - m) is one fma and one approximate base-2 exponent (ex2_fast):
// 2^(x log2 e - m log2 e).
#include <algorithm>
#include <math.h>

#include "ln_device.cuh"
#include "ln_internal.h"

namespace lnk {
namespace {

constexpr int kXeThreads = 512;
constexpr int kXeBlocksPerSm = 3;  // resident blocks: at most 40 registers a thread
constexpr int kXeUnroll = 4;  // 128-bit loads in flight per thread in each pass
constexpr float kLog2e = 1.4426950408889634f;

struct XeParams {
    const void* x;
    const int* targets;
    int rows;
    int V;
    float alpha;
    float dloss;
    float* losses;
    void* dx;
};

// exp(x - m) = 2^(x log2 e + nm) with nm = -m log2 e: one fma and one ex2.
__device__ __forceinline__ float ex_shift(float x, float nm) { return ex2_fast(fmaf(x, kLog2e, nm)); }

// (m, s) += (mb, sb): s sums exp(value - m); a pair with m = -inf holds nothing.
__device__ __forceinline__ void xe_merge(float& m, float& s, float mb, float sb) {
    const float mm = fmaxf(m, mb);
    s = mm == -INFINITY ? 0.f
                        : __fadd_rn(__fmul_rn(s, ex2_fast((m - mm) * kLog2e)),
                                    __fmul_rn(sb, ex2_fast((mb - mm) * kLog2e)));
    m = mm;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kXeThreads, kXeBlocksPerSm) xent_kernel(const XeParams p) {
    using IO = Io<T>;
    using PR = Pairs<T>;
    constexpr int V8 = IO::kVec;
    constexpr int H = PR::kPairs;
    constexpr int NW = kXeThreads / 32;
    __shared__ float red[3][NW];
    __shared__ float xt_sh;
    pdl_enter();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = p.V;
    const T* X = static_cast<const T*>(p.x);
    T* DX = static_cast<T*>(p.dx);
    const float inv_v = 1.0f / (float)V;
    const f2 l2e2 = f2_splat(kLog2e);
    for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const size_t base = (size_t)row * V;
        const int t = p.targets[row];
        if (tid == 0) xt_sh = (t >= 0 && t < V) ? IO::to_f(X[base + t]) : __int_as_float(0x7fc00000);
        // Pass 1: this thread's online (max, sum) pair and plain sum, the sums as even/odd
        // column pairs.
        float m = -INFINITY;
        f2 s2 = f2_splat(0.f), sx2 = f2_splat(0.f);
        if constexpr (VEC) {
            const int nvec = V / V8;
            const uint4* xv = reinterpret_cast<const uint4*>(X + base);
            for (int v0 = tid; v0 < nvec; v0 += kXeUnroll * kXeThreads) {
                uint4 u[kXeUnroll];
#pragma unroll
                for (int k = 0; k < kXeUnroll; ++k) {
                    const int v = v0 + k * kXeThreads;
                    u[k] = v < nvec ? __ldcg(xv + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int k = 0; k < kXeUnroll; ++k) {
                    if (v0 + k * kXeThreads >= nvec) continue;
                    f2 x2[H];
                    PR::unpack(u[k], x2);
                    float mv = fmaxf(f2_lo(x2[0]), f2_hi(x2[0]));
#pragma unroll
                    for (int h = 1; h < H; ++h) mv = fmaxf(mv, fmaxf(f2_lo(x2[h]), f2_hi(x2[h])));
                    if (mv > m) {  // a new running maximum: rescale the sum
                        s2 = m == -INFINITY ? f2_splat(0.f)
                                            : f2_mul(s2, f2_splat(ex2_fast((m - mv) * kLog2e)));
                        m = mv;
                    }
                    if (m != -INFINITY) {
                        const f2 nm2 = f2_splat(-m * kLog2e);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const f2 z = f2_fma(x2[h], l2e2, nm2);
                            s2 = f2_add(s2, f2_make(ex2_fast(f2_lo(z)), ex2_fast(f2_hi(z))));
                        }
                    }
#pragma unroll
                    for (int h = 0; h < H; ++h) sx2 = f2_add(sx2, x2[h]);
                }
            }
        } else {
            float s = 0.f, sx = 0.f;
            for (int j = tid; j < V; j += kXeThreads) {
                const float f = IO::to_f(X[base + j]);
                if (f > m) {
                    s = m == -INFINITY ? 0.f : s * ex2_fast((m - f) * kLog2e);
                    m = f;
                }
                if (m != -INFINITY) s += ex_shift(f, -m * kLog2e);
                sx += f;
            }
            s2 = f2_make(s, 0.f);
            sx2 = f2_make(sx, 0.f);
        }
        float s = f2_lo(s2) + f2_hi(s2), sx = f2_lo(sx2) + f2_hi(sx2);
        // One block reduction of (max, sum) and the plain sum.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float mb = __shfl_xor_sync(kFullMask, m, o);
            const float sb = __shfl_xor_sync(kFullMask, s, o);
            xe_merge(m, s, mb, sb);
            sx += __shfl_xor_sync(kFullMask, sx, o);
        }
        if (lane == 0) {
            red[0][warp] = m;
            red[1][warp] = s;
            red[2][warp] = sx;
        }
        __syncthreads();
        m = red[0][0];
        s = red[1][0];
        sx = red[2][0];
        for (int w = 1; w < NW; ++w) {
            xe_merge(m, s, red[0][w], red[1][w]);
            sx += red[2][w];
        }
        if (tid == 0 && p.losses)
            p.losses[row] = logf(s) + m - ((1.f - p.alpha) * xt_sh + p.alpha * inv_v * sx);
        // Pass 2: dx = dloss * (exp(x - m) / s - alpha / V) and, at the target, minus
        // dloss * (1 - alpha).
        if (DX) {
            const float c = p.dloss / s;
            const float base_p = p.dloss * p.alpha * inv_v;
            const float hit = p.dloss * (1.f - p.alpha);
            const float nm = -m * kLog2e;
            if constexpr (VEC) {
                const int nvec = V / V8;
                const int tv = (t >= 0 && t < V) ? t / V8 : -1;  // the target's vector
                const uint4* xv = reinterpret_cast<const uint4*>(X + base);
                uint4* dv = reinterpret_cast<uint4*>(DX + base);
                const f2 nm2 = f2_splat(nm), c2 = f2_splat(c), nb2 = f2_splat(-base_p);
                for (int v0 = tid; v0 < nvec; v0 += kXeUnroll * kXeThreads) {
                    uint4 u[kXeUnroll];
#pragma unroll
                    for (int k = 0; k < kXeUnroll; ++k) {
                        const int v = v0 + k * kXeThreads;
                        u[k] = v < nvec ? __ldcs(xv + v) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int k = 0; k < kXeUnroll; ++k) {
                        const int v = v0 + k * kXeThreads;
                        if (v >= nvec) continue;
                        f2 x2[H], o[H];
                        PR::unpack(u[k], x2);
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const f2 z = f2_fma(x2[h], l2e2, nm2);
                            o[h] = f2_fma(f2_make(ex2_fast(f2_lo(z)), ex2_fast(f2_hi(z))), c2, nb2);
                        }
                        if (v == tv) {
                            const int ti = t - v * V8;
#pragma unroll
                            for (int h = 0; h < H; ++h)
                                o[h] = f2_sub(o[h], f2_make(2 * h == ti ? hit : 0.f, 2 * h + 1 == ti ? hit : 0.f));
                        }
                        __stcs(dv + v, PR::pack(o));
                    }
                }
            } else {
                for (int j = tid; j < V; j += kXeThreads) {
                    float g = fmaf(ex_shift(IO::to_f(X[base + j]), nm), c, -base_p);
                    if (j == t) g -= hit;
                    DX[base + j] = IO::from_f(g);
                }
            }
        }
        __syncthreads();  // `red` and xt_sh are reused by the next row
    }
}

template <typename T>
cudaError_t launch_xent_t(const XeParams& p, bool vec, cudaStream_t stream) {
    const void* kern = vec ? (const void*)xent_kernel<T, true> : (const void*)xent_kernel<T, false>;
    const DeviceInfo& di = device_info(-1);
    const int occ = std::max(1, blocks_per_sm(kern, kXeThreads, 0));
    const int grid = std::max(1, std::min(p.rows, di.sms * occ));
    XeParams q = p;
    void* args[] = {&q};
    return launch_kernel(kern, dim3(grid), dim3(kXeThreads), 0, stream, args, false);
}

}  // namespace

cudaError_t launch_xent(Dtype dt, const XentArgs& a, bool aligned, cudaStream_t stream,
                        int* launches) {
    *launches = 0;
    if (a.rows == 0) return cudaSuccess;
    XeParams p;
    p.x = a.logits;
    p.targets = a.targets;
    p.rows = a.rows;
    p.V = a.V;
    p.alpha = a.alpha;
    p.dloss = a.dloss;
    p.losses = a.losses;
    p.dx = a.dlogits;
    cudaError_t e = dt == Dtype::F32 ? launch_xent_t<float>(p, aligned, stream)
                                     : launch_xent_t<__nv_bfloat16>(p, aligned, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
