// dropout_rng.h -- the counter-based generator behind the dropout masks, shared by the
// prologue-fused LayerNorm forward and the prologue's backward (host: the round keys;
// device: the words and keep decisions).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lnk {

// ---------------------------------------------------------------------------------------
// Dropout masks from the counter-based generator Philox-4x32 with 10 rounds (Salmon,
// Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011), written
// from the paper's definition.  Element i of a [rows, cols] tensor takes word i % 4 of the
// generator at counter (i / 4, offset) under key `seed`, and is kept when that word is at
// least `thr` = floor(p 2^32): dropped with probability p, and the same mask whenever the
// same (seed, offset) is given again (the backward regenerates it instead of storing it).
//
// One round maps the counter (c0, c1, c2, c3) under round key (k0, k1) to
//   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57, each product taken as one 32 x 32 -> 64-bit multiply;
// the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85) between rounds.  The ten
// round keys depend only on the seed, so they are formed once on the host and travel in the
// kernel parameters, where they are read as constant operands.
// ---------------------------------------------------------------------------------------
struct DropoutRng {
    uint32_t ctr2, ctr3;  // the counter's words 2 and 3: the offset's low and high halves
    uint32_t thr;         // keep when the word is >= thr
    uint32_t k0[10], k1[10];

    static __host__ __device__ DropoutRng make(unsigned long long seed, unsigned long long offset,
                                               uint32_t thr) {
        DropoutRng g;
        g.ctr2 = (uint32_t)offset;
        g.ctr3 = (uint32_t)(offset >> 32);
        g.thr = thr;
        uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
        for (int r = 0; r < 10; ++r) {
            g.k0[r] = a;
            g.k1[r] = b;
            a += 0x9E3779B9u;
            b += 0xBB67AE85u;
        }
        return g;
    }

    // The generator's four words at counter (blk, offset): elements 4 blk .. 4 blk + 3.
    __device__ __forceinline__ uint4 words(unsigned long long blk) const {
        uint4 c = make_uint4((uint32_t)blk, (uint32_t)(blk >> 32), ctr2, ctr3);
#pragma unroll
        for (int r = 0; r < 10; ++r) {
            const unsigned long long p0 = (unsigned long long)c.x * 0xD2511F53u;
            const unsigned long long p1 = (unsigned long long)c.z * 0xCD9E8D57u;
            c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0[r], (uint32_t)p1,
                           (uint32_t)(p0 >> 32) ^ c.w ^ k1[r], (uint32_t)p0);
        }
        return c;
    }
    __device__ __forceinline__ bool keep(unsigned long long i) const {
        const uint4 w = words(i >> 2);
        const uint32_t k = (i & 2) ? ((i & 1) ? w.w : w.z) : ((i & 1) ? w.y : w.x);
        return k >= thr;
    }
};

}  // namespace lnk
