// Counter-based uniforms on the device: Philox4x32 with 10 rounds, written
// from Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1,
// 2, 3" (SC'11).  One block per decision: key = (seed low word, seed high
// word), counter = (b, position, slot, 0); the uniform is the top 24 bits of
// output word 0 scaled by 2^-24, so it lies on the grid {0, 2^-24, ...,
// 1 - 2^-24} and is exact in fp32.
#pragma once

#include <cstdint>

namespace spec {

__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, uint32_t b, uint32_t position,
                                                 uint32_t slot) {
  uint32_t x0 = b, x1 = position, x2 = slot, x3 = 0u;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    // round r uses the key advanced r times by the Weyl increments
    const uint32_t lo_a = 0xD2511F53u * x0, hi_a = __umulhi(0xD2511F53u, x0);
    const uint32_t lo_b = 0xCD9E8D57u * x2, hi_b = __umulhi(0xCD9E8D57u, x2);
    const uint32_t y0 = hi_b ^ x1 ^ k0;
    const uint32_t y2 = hi_a ^ x3 ^ k1;
    x0 = y0;
    x1 = lo_b;
    x2 = y2;
    x3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return x0;
}

__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t b, uint32_t position,
                                                uint32_t slot) {
  return static_cast<float>(philox_word0(seed, b, position, slot) >> 8) * 0x1p-24f;
}

}  // namespace spec
