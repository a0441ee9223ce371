// xent.cu -- fused cross-entropy with label smoothing, forward and backward in one kernel
// (two forms: rows staged whole in shared memory, and rows streamed twice through L2).
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
    unsigned* status;  // the per-device status word (the staged kernel's bounded waits)
    uint64_t limit_ns;
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

// ---------------------------------------------------------------------------------------
// Rows staged in shared memory.  For rows of 16-byte vectors small enough that two fit in
// shared memory (bf16 up to ~56K logits), one persistent 512-thread block per SM keeps two
// row slots filled by 1-D bulk copies (TMA) on mbarriers -- the next row lands while the
// current one is processed -- and makes three passes over the staged row: the maximum m
// (on the raw values: a packed bf16 max per pair), then sum exp(x - m) together with
// sum x, then the gradient.  Each row is read from HBM once, with no online rescaling.
// ---------------------------------------------------------------------------------------
constexpr int kXsThreads = 512;
constexpr int kXsWarps = kXsThreads / 32;

__device__ __forceinline__ float xs_block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kXsWarps; ++w) m = fmaxf(m, red[w]);
    return m;
}

// Two block sums, added in the same order in every thread.
__device__ __forceinline__ void xs_block_sum2(float& a, float& b, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(kFullMask, a, o);
        b += __shfl_xor_sync(kFullMask, b, o);
    }
    if (lane == 0) {
        red[warp] = a;
        red[kXsWarps + warp] = b;
    }
    __syncthreads();
    a = 0.f;
    b = 0.f;
#pragma unroll
    for (int w = 0; w < kXsWarps; ++w) {
        a += red[w];
        b += red[kXsWarps + w];
    }
}

// The largest of a 16-byte vector's values, in fp32 (exact: the I/O values are fp32 or bf16).
template <typename T>
__device__ __forceinline__ float vec_max(const uint4& u) {
    if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 a, b, c, d;
        memcpy(&a, &u.x, 4);
        memcpy(&b, &u.y, 4);
        memcpy(&c, &u.z, 4);
        memcpy(&d, &u.w, 4);
        const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return fmaxf(__low2float(m), __high2float(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                     fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
    }
}

template <typename T>
__global__ void __launch_bounds__(kXsThreads, 1) xent_smem_kernel(const XeParams p, int slot_bytes) {
    using IO = Io<T>;
    using PR = Pairs<T>;
    constexpr int V8 = IO::kVec;
    constexpr int H = PR::kPairs;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t full_bar[2];
    __shared__ float red[2 * kXsWarps];
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const int V = p.V, nvec = V / V8;
    const unsigned row_bytes = (unsigned)V * (unsigned)sizeof(T);
    const T* X = static_cast<const T*>(p.x);
    T* DX = static_cast<T*>(p.dx);
    const float inv_v = 1.0f / (float)V;
    const f2 l2e2 = f2_splat(kLog2e);
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int nmy = b < p.rows ? (p.rows - 1 - b) / G + 1 : 0;
    if (tid == 0) {
        mbar_init(&full_bar[0], 1);
        mbar_init(&full_bar[1], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter();
    auto issue = [&](int k) {  // thread 0: row k of this block into slot k & 1
        if (k >= nmy) return;
        const int row = b + k * G;
        uint64_t* bar = &full_bar[k & 1];
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_g2s(smem_raw + (size_t)(k & 1) * slot_bytes, X + (size_t)row * V, row_bytes, bar);
    };
    if (tid == 0) {
        issue(0);
        issue(1);
    }
    int k = 0;
    for (; k < nmy; ++k) {
        const int row = b + k * G;
        const size_t base = (size_t)row * V;
        const int t = p.targets[row];
        if (!mbar_wait(&full_bar[k & 1], (unsigned)(k >> 1) & 1u, p.limit_ns)) abort_flag = 1;
        __syncthreads();
        if (abort_flag) break;
        const uint4* xs = reinterpret_cast<const uint4*>(smem_raw + (size_t)(k & 1) * slot_bytes);
        // Pass 1: the row maximum.
        float m = -INFINITY;
        // (Each vector is copied to registers with one 128-bit load before use: read through a
        // reference, it would be four 32-bit loads at a 16-byte stride, each 4-way conflicted.)
        for (int v = tid; v < nvec; v += kXsThreads) {
            const uint4 u = xs[v];
            m = fmaxf(m, vec_max<T>(u));
        }
        m = xs_block_max(m, red);
        // Pass 2: sum exp(x - m) and sum x (even/odd column pairs).
        const float nm = m == -INFINITY ? 0.f : -m * kLog2e;
        const f2 nm2 = f2_splat(nm);
        f2 s2 = f2_splat(0.f), sx2 = f2_splat(0.f);
        for (int v = tid; v < nvec; v += kXsThreads) {
            const uint4 u = xs[v];
            f2 x2[H];
            PR::unpack(u, x2);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const f2 z = f2_fma(x2[h], l2e2, nm2);
                s2 = f2_add(s2, f2_make(ex2_fast(f2_lo(z)), ex2_fast(f2_hi(z))));
                sx2 = f2_add(sx2, x2[h]);
            }
        }
        float s = f2_lo(s2) + f2_hi(s2), sx = f2_lo(sx2) + f2_hi(sx2);
        __syncthreads();  // `red` is reused
        xs_block_sum2(s, sx, red);
        if (tid == 0 && p.losses) {
            const float xt = (t >= 0 && t < V)
                                 ? IO::to_f(reinterpret_cast<const T*>(xs)[t])
                                 : __int_as_float(0x7fc00000);
            p.losses[row] = logf(s) + m - ((1.f - p.alpha) * xt + p.alpha * inv_v * sx);
        }
        // Pass 3: dx = dloss * (exp(x - m) / s - alpha / V), minus dloss * (1 - alpha) at the
        // target.
        if (DX) {
            const float c = p.dloss / s;
            const float base_p = p.dloss * p.alpha * inv_v;
            const float hit = p.dloss * (1.f - p.alpha);
            const int tv = (t >= 0 && t < V) ? t / V8 : -1;
            const f2 c2 = f2_splat(c), nb2 = f2_splat(-base_p);
            uint4* dv = reinterpret_cast<uint4*>(DX + base);
            for (int v = tid; v < nvec; v += kXsThreads) {
                const uint4 u = xs[v];
                f2 x2[H], o[H];
                PR::unpack(u, x2);
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
        __syncthreads();  // every thread is done with the slot and with `red`
        if (tid == 0) issue(k + 2);
    }
    if (abort_flag) {
        if (tid == 0) {
            raise_status(p.status, kStatusTimeout);
            for (int j = k; j < k + 2 && j < nmy; ++j)  // drain: the copies still in flight
                (void)mbar_wait(&full_bar[j & 1], (unsigned)(j >> 1) & 1u, p.limit_ns);
        }
        __syncthreads();
    }
}

// Bytes of one row slot: the row rounded up to a multiple of 128.
inline int xent_slot_bytes(int V, size_t esize) { return (int)(((size_t)V * esize + 127) / 128 * 128); }

template <typename T>
cudaError_t launch_xent_t(const XeParams& p, bool vec, cudaStream_t stream) {
    const DeviceInfo& di = device_info(-1);
    XeParams q = p;
    void* args[] = {&q};
    const int slot = xent_slot_bytes(p.V, sizeof(T));
    const size_t smem = 2 * (size_t)slot;
    if (vec && smem + 1024 <= (size_t)di.smem_optin) {  // two staged rows fit: one HBM read
        const void* kern = (const void*)xent_smem_kernel<T>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int slot_arg = slot;
        void* sargs[] = {&q, &slot_arg};
        const int grid = std::max(1, std::min(p.rows, di.sms));
        return launch_kernel(kern, dim3(grid), dim3(kXsThreads), smem, stream, sargs, false);
    }
    const void* kern = vec ? (const void*)xent_kernel<T, true> : (const void*)xent_kernel<T, false>;
    const int occ = std::max(1, blocks_per_sm(kern, kXeThreads, 0));
    const int grid = std::max(1, std::min(p.rows, di.sms * occ));
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
    p.status = a.status;
    p.limit_ns = a.wait_limit_ns;
    cudaError_t e = dt == Dtype::F32 ? launch_xent_t<float>(p, aligned, stream)
                                     : launch_xent_t<__nv_bfloat16>(p, aligned, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace lnk
