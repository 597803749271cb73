// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11, section 3) and the noise transforms of the
// draft step: a request's 64-bit seed is the key (lo32, hi32), the counter names
// (column / 4, position, domain, step).
#pragma once

#include <stdint.h>

namespace fm {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;  // Weyl key increments of the paper
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ uint4 philox_seeded(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return philox4x32_10(make_uint4(c0, c1, c2, c3), static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

// U = ((w >> 9) + 1/2) * 2^-23: exact in float32, strictly inside (0, 1).
__device__ __forceinline__ float word_to_uniform(uint32_t w) {
  return (static_cast<float>(w >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

// Box-Muller: (r cos 2 pi Ub, r sin 2 pi Ub), r = sqrt(-2 ln Ua).
__device__ __forceinline__ float2 box_muller(uint32_t wa, uint32_t wb) {
  const float ua = word_to_uniform(wa), ub = word_to_uniform(wb);
  const float r = sqrtf(-2.f * logf(ua));
  float s, c;
  sincospif(2.f * ub, &s, &c);
  return make_float2(r * c, r * s);
}

// Gumbel noise -ln(-ln U).
__device__ __forceinline__ float gumbel_of_word(uint32_t w) { return -logf(-logf(word_to_uniform(w))); }

constexpr uint32_t kDomainDraftNoise = 0;
constexpr uint32_t kDomainGumbel = 1;

}  // namespace fm
