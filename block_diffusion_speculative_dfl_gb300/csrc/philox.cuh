// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror & Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), the one device copy
// every kernel that draws a uniform uses.
//
// One round multiplies counter words 0 and 2 by the round multipliers
// (32x32 -> 64 bits); the new counter is (hi(c2 m1) ^ c1 ^ k0, lo(c2 m1),
// hi(c0 m0) ^ c3 ^ k1, lo(c0 m0)); the key advances by the Weyl constants
// between rounds.  Ten rounds.
#pragma once

#include <stdint.h>

namespace dfl {

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
    #pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// The uniform of counter (c0, c1, c2, c3) and key (k0, k1): the top 24 bits
// of output word 0, u = ((x0 >> 8) + 1/2) 2^-24, strictly inside (0, 1) and
// exact in fp64.
__device__ __forceinline__ double philox_uniform24(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                   uint32_t k1) {
    const uint32_t x0 = philox4x32_10(c0, c1, c2, c3, k0, k1).x;
    return ((double)(x0 >> 8) + 0.5) * (1.0 / 16777216.0);
}

}  // namespace dfl
