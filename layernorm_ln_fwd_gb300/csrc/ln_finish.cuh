// ln_finish.cuh -- the second stage of the deterministic column sums, shared by the
// LayerNorm / RMSNorm backward kernels and the dropout backward: blocks that own a slice of
// the columns read every block's partial sums of their slice as they land, add them in a
// fixed order and write the result.  The parameter struct A provides part, cols, nstat,
// fin_rw, status, limit_ns and the outputs dgamma (statistic 0) and dbeta (statistic 1).
#pragma once

#include <climits>

#include "ln_device.cuh"

namespace lnk {
namespace {

// (S, C) += (h, l), where a compensated value is S + C.
__device__ __forceinline__ void comp_add(float& S, float& C, float h, float l) {
    float s, e;
    two_sum_f(S, h, s, e);
    S = s;
    C += e + l;
}

// ---------------------------------------------------------------------------------------
// Stage 2: the finish.  A unit is U adjacent columns of one statistic; a partial is a
// (hi, lo) pair per column, or one plain fp32 sum when COMPACT, and U is chosen so that one
// unit of one partial row is a single 16-byte load where the row length allows.  Units are
// taken in groups of kFinUnits adjacent ones (128 contiguous bytes of a partial row); block f
// of the F finishing blocks owns groups [f * g / F, (f + 1) * g / F).  The block's warps work on GW groups at a
// time, RW warps per group (RW * GW = the warp count, RW chosen by the host so that a lane's
// rows fit in one batch).  Warp r of a group's RW takes the contiguous range of partial rows
// [r * P / RW, (r + 1) * P / RW); lane (s, k), s < kFinSub, k < kFinUnits, adds unit k of
// rows s, s + kFinSub, ... of that range in increasing order (the loads of a batch issued
// before the first addition, so the L2 latency is paid once per batch, and a warp's load
// touches kFinSub lines); the kFinSub lane totals are folded by a fixed shuffle tree, and
// the RW warp totals are added in warp order through shared memory.  The order depends
// only on P, RW and the unit.
// A loaded unit with a zero word belongs to a block that has not written its partials yet:
// one lane of the warp watches a single word of the earliest such row, the lanes then reload
// what they miss, until nothing is missing or the time limit passes; then each lane zeroes
// the units it read and adds them.
// Compensated partials are added with TwoSum; COMPACT partials (plain fp32 sums from
// kernels with bf16 results) with plain fp32 additions: their error, about 2^-24 * sqrt(P)
// times the partials' size, is far below a bf16 unit in the last place.
// `scratch` holds at least 2 * U floats per thread.
// ---------------------------------------------------------------------------------------
constexpr int kFinUnits = 8;
constexpr int kFinSub = 32 / kFinUnits;
constexpr int kFinBatch = 48;  // at most this many words of partials per lane and batch,
constexpr int kFinMaxRows = 10;  // from at most this many partial rows
__host__ __device__ constexpr int fin_rows_per_lane(int words_per_unit) {
    return kFinBatch / words_per_unit < kFinMaxRows ? kFinBatch / words_per_unit : kFinMaxRows;
}

// The same pointer, opaque to the compiler (so values derived from it are recomputed, not
// kept live from an earlier computation).
template <typename P>
__device__ __forceinline__ P* opaque(P* p) {
    asm volatile("" : "+l"(p));
    return p;
}

template <int N>
__device__ __forceinline__ bool has_zero(const uint32_t (&w)[N]) {
    bool z = false;
#pragma unroll
    for (int i = 0; i < N; ++i) z |= w[i] == 0u;
    return z;
}

template <typename T, int U, bool COMPACT, typename A>
__device__ void finish_units(const A& a, int P, int F, int f, float* scratch) {
    using IO = Io<T>;
    constexpr int E = COMPACT ? 1 : 2;  // floats per column of a partial
    constexpr int W = E * U;            // words per unit of a partial row: 1, 2 or 4
    constexpr int L = fin_rows_per_lane(W);  // partial rows one lane loads per batch
    const int cols = a.cols;
    const int ngroups = cols / U;       // units per statistic
    const int nunits = a.nstat * ngroups;
    const int ng = (nunits + kFinUnits - 1) / kFinUnits;
    const int g0 = f * ng / F, g1 = (f + 1) * ng / F;  // f * ng < 2^24: 32-bit is exact
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int RW = a.fin_rw, GW = nw / RW;
    const int gw = warp / RW, rw = warp - gw * RW;
    const int k = lane % kFinUnits, sub = lane / kFinUnits;
    const int p_lo = rw * P / RW, p_hi = (rw + 1) * P / RW;
    uint32_t* part = reinterpret_cast<uint32_t*>(a.part);
    const size_t stat_stride = (size_t)P * cols * E;
    const size_t row_stride = (size_t)cols * E;
    bool late = false;  // a partial did not arrive within the time limit
    for (int gb = g0; gb < g1; gb += GW) {  // block-uniform
        const int gi = gb + gw;
        const int u = gi * kFinUnits + k;
        const bool grp_ok = gi < g1;  // the same in the whole warp
        const bool act = grp_ok && u < nunits;
        const int stat = u >= ngroups ? 1 : 0, grp = u - stat * ngroups;
        float S[U], C[U];
#pragma unroll
        for (int i = 0; i < U; ++i) S[i] = C[i] = 0.f;
        if (grp_ok) {
            uint32_t* src = part + stat * stat_stride + (size_t)grp * W;
            const size_t step = (size_t)kFinSub * row_stride;  // between a lane's rows
            for (int pb = p_lo; pb < p_hi; pb += kFinSub * L) {  // the same trips in the warp
                const int p0 = pb + sub;
                const int nj = act && p0 < p_hi ? (p_hi - p0 + kFinSub - 1) / kFinSub : 0;
                uint32_t* q0 = src + (size_t)p0 * row_stride;
                uint32_t v[L][W];
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    if (j < nj) {
                        ld_part<W>(q0 + j * step, v[j]);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[j][i] = ~0u;  // reads as +0
                    }
                }
                unsigned miss = 0;  // bit j: row j of this lane's batch is not all there
#pragma unroll
                for (int j = 0; j < L; ++j) miss |= has_zero<W>(v[j]) ? 1u << j : 0u;
                if (__any_sync(kFullMask, miss != 0)) {
                    // Blocks still writing.  Lane 0 watches one word (its unit) of the warp's
                    // earliest missing row until it is written -- one load per warp and
                    // round, not one per missing unit -- then the lanes reload what they
                    // miss, until nothing is missing or the time limit passes.
                    const uint64_t t0 = global_ns();
                    while (true) {
                        const int mine = miss ? p0 + (__ffs((int)miss) - 1) * kFinSub : INT_MAX;
                        const int pw = __reduce_min_sync(kFullMask, mine);
                        if (pw == INT_MAX) break;
                        int gave_up = 0;
                        if (lane == 0) {  // lane 0 owns unit 0 of the group, which exists
                            const uint32_t* wq = opaque(src) + (size_t)pw * row_stride;
                            uint32_t w1[1];
                            ld_part<1>(wq, w1);
                            while (w1[0] == 0u) {
                                if (global_ns() - t0 > a.limit_ns) {
                                    gave_up = 1;
                                    break;
                                }
                                __nanosleep(128);
                                ld_part<1>(wq, w1);
                            }
                        }
                        if (__shfl_sync(kFullMask, gave_up, 0)) {
                            late = true;
                            break;
                        }
                        const uint32_t* q = opaque(q0);  // addresses recomputed, not kept live
#pragma unroll
                        for (int j = 0; j < L; ++j)
                            if (miss & (1u << j)) ld_part<W>(q + j * step, v[j]);
                        miss = 0;
#pragma unroll
                        for (int j = 0; j < L; ++j) miss |= has_zero<W>(v[j]) ? 1u << j : 0u;
                    }
                }
                uint32_t* qz = opaque(q0);
#pragma unroll
                for (int j = 0; j < L; ++j)  // read: cleared for the next call
                    if (j < nj) st_zero<W>(qz + j * step);
#pragma unroll
                for (int j = 0; j < L; ++j)
#pragma unroll
                    for (int i = 0; i < U; ++i) {
                        if constexpr (COMPACT)
                            S[i] += part_dec(v[j][i]);
                        else
                            comp_add(S[i], C[i], part_dec(v[j][2 * i]), part_dec(v[j][2 * i + 1]));
                    }
            }
        }
        // Fold the row subsets: lane (s, k) takes in lane (s + o, k) for o = 2, 1 (in units
        // of kFinUnits lanes); lane (0, k) ends with the warp's total of unit k.
#pragma unroll
        for (int o = kFinSub / 2; o > 0; o >>= 1) {
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const float s2 = __shfl_down_sync(kFullMask, S[i], o * kFinUnits);
                const float c2 = __shfl_down_sync(kFullMask, C[i], o * kFinUnits);
                if constexpr (COMPACT)
                    S[i] += s2;
                else
                    comp_add(S[i], C[i], s2, c2);
            }
        }
        if (sub == 0) {
            float* mine = scratch + ((size_t)warp * kFinUnits + k) * 2 * U;
#pragma unroll
            for (int i = 0; i < U; ++i) {
                mine[2 * i] = S[i];
                mine[2 * i + 1] = C[i];
            }
        }
        __syncthreads();
        if (rw == 0 && sub == 0 && act) {  // the group's warp totals, in warp order
            float T2[U], C2[U];
#pragma unroll
            for (int i = 0; i < U; ++i) T2[i] = C2[i] = 0.f;
            for (int w = warp; w < warp + RW; ++w) {
                const float* o = scratch + ((size_t)w * kFinUnits + k) * 2 * U;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    if constexpr (COMPACT)
                        T2[i] += o[2 * i];
                    else
                        comp_add(T2[i], C2[i], o[2 * i], o[2 * i + 1]);
                }
            }
            T* dst = static_cast<T*>(stat == 0 ? a.dgamma : a.dbeta) + (size_t)grp * U;
#pragma unroll
            for (int i = 0; i < U; ++i) dst[i] = IO::from_f(T2[i] + C2[i]);
        }
        __syncthreads();  // scratch is reused by the next group
    }
    if (late) raise_status(a.status, kStatusTimeout);
}

// Warps per unit group in the finish: the fewest (a divisor of the block's nw warps) for
// which one batch of loads per lane covers all P partial rows, with W words per unit.
inline int fin_warps_per_group(int nw, int P, int words_per_unit) {
    const int rows_per_warp_batch = kFinSub * fin_rows_per_lane(words_per_unit);
    const int need = (P + rows_per_warp_batch - 1) / rows_per_warp_batch;
    for (int d = 1; d <= nw; ++d)
        if (nw % d == 0 && d >= need) return d;
    return nw;
}

}  // namespace
}  // namespace lnk
