// The verifier's uniforms: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11), keyed by the seed and counted by (row, position).
#pragma once

#include <stdint.h>

namespace mtpspec {

// Ten rounds of two 32x32->64 multiplications with the round multipliers, half swaps and
// key mixing; the key advances by the two Weyl increments after each round.
__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}
// odd multiple of 2^-24 in (0, 1), exact in fp32
__device__ __forceinline__ float word_uniform(uint32_t w) {
    return __uint2float_rn(2u * (w >> 9) + 1u) * 5.9604644775390625e-08f;
}
// U_acc (word 0) and U_smp (word 1) of unit (row, position)
__device__ __forceinline__ void unit_uniforms(uint64_t seed, uint32_t row, uint32_t pos,
                                              float &u_acc, float &u_smp) {
    uint32_t c[4] = {row, pos, 0u, 0u};
    philox(c, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    u_acc = word_uniform(c[0]);
    u_smp = word_uniform(c[1]);
}

}  // namespace mtpspec
