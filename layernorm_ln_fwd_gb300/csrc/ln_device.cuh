// ln_device.cuh -- device-side building blocks shared by the forward and backward kernels.
//
// 128-bit vectors of the I/O type and their fp32-pair forms, warp reductions, row shifts and
// mergeable row statistics, bulk-copy (TMA) staging with mbarriers and ring positions, the
// programmatic-dependent-launch entry, bounded waits and the per-device status word.
// Everything here is sm_100-family code (built for sm_103a); nothing here allocates.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dropout_rng.h"

namespace lnk {

constexpr unsigned kFullMask = 0xffffffffu;

// Bit set in the status word when a bounded wait ran out.
constexpr unsigned kStatusTimeout = 1u;

// ---------------------------------------------------------------------------------------
// I/O element types.  A "vector" is 16 bytes: 4 fp32 or 8 bf16 values.
// ---------------------------------------------------------------------------------------
template <typename T>
struct Io;

template <>
struct Io<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
    // Round an fp32 value to the I/O type and back (identity for fp32).
    static __device__ __forceinline__ float round(float v) { return v; }
    static __device__ __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    // Element-wise a + b of two vectors, rounded to the I/O type.
    static __device__ __forceinline__ uint4 add_round(const uint4& a, const uint4& b) {
        return make_uint4(__float_as_uint(__uint_as_float(a.x) + __uint_as_float(b.x)),
                          __float_as_uint(__uint_as_float(a.y) + __uint_as_float(b.y)),
                          __float_as_uint(__uint_as_float(a.z) + __uint_as_float(b.z)),
                          __float_as_uint(__uint_as_float(a.w) + __uint_as_float(b.w)));
    }
};

template <>
struct Io<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    static __device__ __forceinline__ float round(float v) {
        return __bfloat162float(__float2bfloat16_rn(v));
    }
    static __device__ __forceinline__ float2 pair(uint32_t w) {
        __nv_bfloat162 h;
        memcpy(&h, &w, 4);
        return __bfloat1622float2(h);
    }
    static __device__ __forceinline__ uint32_t pair_bits(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    static __device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
        float2 p0 = pair(u.x), p1 = pair(u.y), p2 = pair(u.z), p3 = pair(u.w);
        f[0] = p0.x; f[1] = p0.y; f[2] = p1.x; f[3] = p1.y;
        f[4] = p2.x; f[5] = p2.y; f[6] = p3.x; f[7] = p3.y;
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
        return make_uint4(pair_bits(f[0], f[1]), pair_bits(f[2], f[3]), pair_bits(f[4], f[5]),
                          pair_bits(f[6], f[7]));
    }
    // Element-wise a + b of two vectors, rounded to bf16: one packed add.rn.bf16x2 per pair.
    // The exact sum of two bf16 values is rounded once, which is the same number as the
    // fp32 sum (exact for two bf16 operands) rounded to bf16.
    static __device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        __nv_bfloat162 x, y;
        memcpy(&x, &a, 4);
        memcpy(&y, &b, 4);
        const __nv_bfloat162 z = __hadd2(x, y);
        uint32_t w;
        memcpy(&w, &z, 4);
        return w;
    }
    static __device__ __forceinline__ uint4 add_round(const uint4& a, const uint4& b) {
        return make_uint4(add2(a.x, b.x), add2(a.y, b.y), add2(a.z, b.z), add2(a.w, b.w));
    }
};

// ---------------------------------------------------------------------------------------
// Packed fp32 pairs.  sm_100-family SMs execute add, sub, mul and fma on two fp32 values
// held in a 64-bit register pair as one instruction (PTX .f32x2).  Each half is an ordinary
// IEEE fp32 operation rounded to nearest even, so a pair computes bit for bit what two
// scalar __fadd_rn / __fmul_rn / fmaf calls would, in half the issue slots.  Nothing is
// contracted across these calls: a product rounded by f2_mul stays rounded.
// ---------------------------------------------------------------------------------------
struct f2 {
    unsigned long long v;
};

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2 f2_splat(float a) { return f2_make(a, a); }
__device__ __forceinline__ float f2_lo(f2 a) {
    float lo;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {%0, t}, %1;\n\t}" : "=f"(lo) : "l"(a.v));
    return lo;
}
__device__ __forceinline__ float f2_hi(f2 a) {
    float hi;
    asm("{\n\t.reg .f32 t;\n\tmov.b64 {t, %0}, %1;\n\t}" : "=f"(hi) : "l"(a.v));
    return hi;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
// a * b + c with one rounding per half.
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return d;
}

// A 16-byte vector as fp32 pairs: element 2h in the low half of pair h, 2h + 1 in the high.
template <typename T>
struct Pairs;

template <>
struct Pairs<float> {
    static constexpr int kPairs = 2;
    static __device__ __forceinline__ void unpack(const uint4& u, f2 (&p)[2]) {
        p[0].v = (unsigned long long)u.x | ((unsigned long long)u.y << 32);
        p[1].v = (unsigned long long)u.z | ((unsigned long long)u.w << 32);
    }
    static __device__ __forceinline__ uint4 pack(const f2 (&p)[2]) {
        return make_uint4((uint32_t)p[0].v, (uint32_t)(p[0].v >> 32), (uint32_t)p[1].v,
                          (uint32_t)(p[1].v >> 32));
    }
    // A vector staged in shared memory, as its two pairs, with ONE 128-bit load.  (Left to
    // itself the compiler reads such a vector as two 64-bit loads, one per pair; at a lane
    // stride of 16 bytes each of those is 2-way bank-conflicted.)  Ordered after the wait
    // that made the data visible, like any other memory access.
    static __device__ __forceinline__ void load_staged(const float* p, f2 (&o)[2]) {
        asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];"
                     : "=l"(o[0].v), "=l"(o[1].v)
                     : "r"((unsigned)__cvta_generic_to_shared(p))
                     : "memory");
    }
};

template <>
struct Pairs<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    // A bf16 value is the upper half of the fp32 value it stands for.
    static __device__ __forceinline__ f2 word(uint32_t w) {
        return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ void unpack(const uint4& u, f2 (&p)[4]) {
        p[0] = word(u.x);
        p[1] = word(u.y);
        p[2] = word(u.z);
        p[3] = word(u.w);
    }
    // Both halves rounded to bf16 (nearest even) into one 32-bit word, low half first.
    static __device__ __forceinline__ uint32_t bits(f2 a) {
        uint32_t w;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(f2_hi(a)), "f"(f2_lo(a)));
        return w;
    }
    static __device__ __forceinline__ uint4 pack(const f2 (&p)[4]) {
        return make_uint4(bits(p[0]), bits(p[1]), bits(p[2]), bits(p[3]));
    }
    // A vector staged in shared memory (one 128-bit load: its four words feed four pairs).
    static __device__ __forceinline__ void load_staged(const __nv_bfloat16* p, f2 (&o)[4]) {
        unpack(*reinterpret_cast<const uint4*>(p), o);
    }
};

// 2^t by the special-function unit's approximate exponent (PTX ex2.approx.ftz.f32: one
// instruction, a few units in the last place; results below 2^-126 flush to zero).  Used
// for softmax weights, where t <= 0 and a flushed term is below 2^-126 of the row's
// largest; the full-range library exp2f costs several instructions more per element.
__device__ __forceinline__ float ex2_fast(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// ---------------------------------------------------------------------------------------
// Global memory access with cache hints.  The row outputs are written once per kernel with
// the evict-first ("cs") policy so they do not push gamma/beta or the backward's partial sums
// out of L2 (the row inputs arrive by bulk copies into shared memory).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_keep(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// ---------------------------------------------------------------------------------------
// Reductions.  The xor butterfly leaves the same bits in every lane: at each step the two
// lanes of a pair add the same two operands, and fp32 addition is commutative.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void warp_sum2(float& a, float& b) {
    f2 v = f2_make(a, b);  // both sums added as one fp32 pair per step
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = f2_add(v, f2_make(__shfl_xor_sync(kFullMask, f2_lo(v), o),
                              __shfl_xor_sync(kFullMask, f2_hi(v), o)));
    a = f2_lo(v);
    b = f2_hi(v);
}

// The sums of n <= 32 per-warp values of two statistics exchanged through shared memory
// (sa[0..n), sb[0..n)), the same bits in every thread of the block: each warp loads them into
// its lanes (zeros past n) and adds them with the xor butterfly -- two loads and five
// shuffle-adds instead of a serial loop over the warps.
__device__ __forceinline__ void sum_warp_values2(const float* sa, const float* sb, int n,
                                                 float& a, float& b) {
    const int lane = threadIdx.x & 31;
    a = lane < n ? sa[lane] : 0.f;
    b = lane < n ? sb[lane] : 0.f;
    warp_sum2(a, b);
}

// Division by the row length without a division per row: with inv = 1/n rounded once per
// kernel, q0 = a * inv rounded, the residual r = a - q0 * n exact in one fma, and one
// correction q = q0 + r * inv give the correctly rounded a / n (Markstein's correction; see
// Muller et al., "Handbook of Floating-Point Arithmetic", on Markstein's theorem), i.e. the
// bits a division would give, in three instructions.
struct RowDivisor {
    float n, inv;
    __device__ explicit RowDivisor(int cols) : n((float)cols), inv(1.0f / (float)cols) {}
    __device__ __forceinline__ float div(float a) const {
        const float q = __fmul_rn(a, inv);
        const float r = __fmaf_rn(-q, n, a);
        return __fmaf_rn(r, inv, q);
    }
};

// Row statistics without E[x^2] - E[x]^2 ("Accelerating Transformer on GPU (I)", section 4.2:
// the pairwise update of Welford and Chan).  Each lane (or thread) summarises its own values
// of a row as a count n, the mean m of d = s - K and the sum M2 of squared deviations of d
// from m, where K is one value of the row shared by all lanes (so the lane means are small
// numbers whenever K is a typical value; M2 does not depend on K at all).  The summaries are
// merged pairwise with
//   n = na + nb,  m = (na ma + nb mb) / n,  M2 = M2a + M2b + (mb - ma)^2 na nb / n,
// a sum of non-negative terms: nothing cancels, whichever value K is.  The merge is written
// in a form symmetric in (a, b) -- separate products, commutative sums, delta^2 -- so both
// lanes of an xor-butterfly pair end with the same bits and, after the butterfly, every lane
// of the warp holds the same summary.  (The section prints the mean update as
// ma + delta nb / n; the weighted form computes the same number and is symmetric.)
//
// The plain sum S of the unshifted values travels with the summary: the stored mean is S / n,
// which carries only the rounding of sums of the row's own values (K + m would carry K's
// distance to the mean times the unit roundoff, large when K is an outlier).
//
// One level of the merge with partner offset o and weights wa = na / n, wb = nb / n,
// w = na nb / n (this lane holds the na-value summary).
__device__ __forceinline__ void chan_step(int o, float wa, float wb, float w, float& S,
                                          float& m, float& M2) {
    const float Sb = __shfl_xor_sync(kFullMask, S, o);
    const float mb = __shfl_xor_sync(kFullMask, m, o);
    const float qb = __shfl_xor_sync(kFullMask, M2, o);
    const float delta = __fsub_rn(mb, m);
    S = __fadd_rn(S, Sb);
    M2 = __fmaf_rn(__fmul_rn(delta, delta), w, __fadd_rn(M2, qb));
    m = __fadd_rn(__fmul_rn(wa, m), __fmul_rn(wb, mb));
}

// Butterfly over xor offsets `first`, first / 2, ..., 1 when every lane's summary covers the
// same count n: each level merges two equal halves (wa = wb = 1/2, w = n / 2, n doubling).
__device__ __forceinline__ void chan_reduce_equal(int first, float n, float& S, float& m,
                                                  float& M2) {
    for (int o = first; o > 0; o >>= 1) {
        chan_step(o, 0.5f, 0.5f, __fmul_rn(n, 0.5f), S, m, M2);
        n = __fadd_rn(n, n);
    }
}

// Butterfly over all 32 lanes for any counts (n = this lane's; 0 for a lane with no values).
__device__ __forceinline__ void chan_reduce_any(float n, float& S, float& m, float& M2) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float nb = __shfl_xor_sync(kFullMask, n, o);
        float wa = 1.f, wb = 0.f, w = 0.f;
        if (n == 0.f) {
            wa = 0.f;
            wb = 1.f;
        } else if (nb != 0.f) {
            const float inv = __frcp_rn(__fadd_rn(n, nb));  // counts are small integers
            wa = __fmul_rn(n, inv);
            wb = __fmul_rn(nb, inv);
            w = __fmul_rn(__fmul_rn(n, nb), inv);
        }
        chan_step(o, wa, wb, w, S, m, M2);
        n = __fadd_rn(n, nb);
    }
}

// The shift K of the scalar kernel's Welford summaries: the median of five of the row's
// stored values, at columns 0, C/4, C/2, 3C/4 and C - 1.  Any K gives the same M2; K only
// sets the size of the shifted values d, whose rounding (when |d| is large next to s) and
// whose mean's rounding reach xhat as about the unit roundoff times |K - mean| * rstd.  The
// median of a spread sample stays within the body of the row whatever a few values (an
// outlier in the first column, say) are.
__device__ __forceinline__ float median5(float a, float b, float c, float d, float e) {
    const float f = fmaxf(fminf(a, b), fminf(c, d));
    const float g = fminf(fmaxf(a, b), fmaxf(c, d));
    return fmaxf(fminf(e, f), fminf(fmaxf(e, f), g));  // the median of (e, f, g)
}

// A vector's first value (the low bf16 of its first word for bf16).
template <typename T>
__device__ __forceinline__ float first_value(const uint4& v) {
    if constexpr (Io<T>::kVec == 8)
        return __uint_as_float(v.x << 16);
    else
        return __uint_as_float(v.x);
}

__device__ __forceinline__ int sample_col(int j, int cols) { return (int)(((long long)j * (cols - 1)) / 4); }

// K from a row held in shared or global memory: s = x + res rounded to the I/O type (or x).
template <typename T, bool HAS_RES>
__device__ __forceinline__ float row_shift(const T* xs, const T* rs, int cols) {
    float v[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        const int c = sample_col(j, cols);
        v[j] = HAS_RES ? Io<T>::round(Io<T>::to_f(xs[c]) + Io<T>::to_f(rs[c])) : Io<T>::to_f(xs[c]);
    }
    return median5(v[0], v[1], v[2], v[3], v[4]);
}

__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// ---------------------------------------------------------------------------------------
// Status word and time.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_status(unsigned* status, unsigned bit) {
    if (status) atomicOr(status, bit);
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------------------------------
// Partial sums that announce themselves.  The backward's per-block partial sums go to a
// workspace whose words are all zero between calls.  A partial is stored as the complement
// of its fp32 bits, the one pattern whose complement is zero (0xffffffff, a NaN) first
// replaced by its neighbour 0xfffffffe (also a NaN), so a stored partial is never the zero
// word and a zero word is one not written yet.  Readers poll with strong (relaxed, GPU-scope)
// loads until none of the words they need is zero, then put zeros back for the next call.
// Every word is written once per call and read whole (aligned 32-bit accesses are
// single-copy atomic), so neither a fence nor a counter is needed to publish the partials.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t part_enc(float x) {
    return ~min(__float_as_uint(x), 0xfffffffeu);
}
__device__ __forceinline__ float part_dec(uint32_t w) { return __uint_as_float(~w); }

__device__ __forceinline__ void st_part4(void* p, float a, float b, float c, float d) {
    asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p),
                 "r"(part_enc(a)), "r"(part_enc(b)), "r"(part_enc(c)), "r"(part_enc(d))
                 : "memory");
}
__device__ __forceinline__ void st_part2(void* p, float a, float b) {
    asm volatile("st.relaxed.gpu.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(part_enc(a)),
                 "r"(part_enc(b))
                 : "memory");
}

// Strong loads of N = 4, 2 or 1 consecutive words (16-, 8- or 4-byte aligned).
template <int N>
__device__ __forceinline__ void ld_part(const void* p, uint32_t (&w)[N]) {
    if constexpr (N == 4)
        asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "l"(p)
                     : "memory");
    else if constexpr (N == 2)
        asm volatile("ld.relaxed.gpu.global.v2.b32 {%0, %1}, [%2];"
                     : "=r"(w[0]), "=r"(w[1])
                     : "l"(p)
                     : "memory");
    else
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(w[0]) : "l"(p) : "memory");
}

template <int N>
__device__ __forceinline__ void st_zero(void* p) {
    if constexpr (N == 4)
        *reinterpret_cast<uint4*>(p) = make_uint4(0u, 0u, 0u, 0u);
    else if constexpr (N == 2)
        *reinterpret_cast<uint2*>(p) = make_uint2(0u, 0u);
    else
        *reinterpret_cast<uint32_t*>(p) = 0u;
}

// Wait until *ctr >= target or `limit_ns` has passed.  Returns whether the target was seen.
__device__ __forceinline__ bool wait_counter_geq(const unsigned* ctr, unsigned target,
                                                 uint64_t limit_ns) {
    if (ld_acquire_u32(ctr) >= target) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire_u32(ctr) >= target) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------------------
// Bulk copies (TMA, non-tensor form) global -> shared, completed on an mbarrier.
// Source and destination must be 16-byte aligned and the size a multiple of 16.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Test the phase with the given parity; a thread whose phase is not complete yet is
// suspended in hardware until it completes or about `hint_ns` have passed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity, unsigned hint_ns) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  The suspend hint keeps a
// waiting warp off the issue slots; the time limit is checked between suspensions.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, uint64_t limit_ns) {
    constexpr unsigned kHintNs = 100000;
    if (mbar_try_wait(bar, parity, kHintNs)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity, kHintNs)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Position in a ring of n slots: the slot index and the parity of the current pass over the
// ring (the mbarrier phase parity a waiter on that slot needs), advanced without division.
struct RingPos {
    int slot = 0;
    unsigned phase = 0;
    __device__ __forceinline__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Programmatic dependent launch (the kernels are launched with programmatic stream
// serialization allowed).  Before its first access to global memory (its shared-memory
// set-up may come first) a kernel waits until the grid before it in the stream has completed
// and its memory is visible (a no-op when there is none), then lets the grid after it begin
// launching: that grid's blocks take SMs as this grid's blocks leave and do their own set-up,
// but they too wait here before touching global memory, so stream order holds.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Default limit of every device-side wait: 2 seconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

}  // namespace lnk
