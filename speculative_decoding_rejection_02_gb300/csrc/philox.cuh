// Device Philox4x32-10 and the verifier's two uniform constructions.
//
// Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and
// Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of
// two 32x32->64 multiplies by the published constants, a word crossing and a
// key mix, with the key advanced by the published Weyl increments between
// rounds. Written here for the device from that definition.
#pragma once
#include <cstdint>

namespace sv {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t a = c.x, b = c.z;
    const uint32_t hi0 = __umulhi(0xD2511F53u, a), lo0 = 0xD2511F53u * a;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, b), lo1 = 0xCD9E8D57u * b;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

constexpr uint32_t kTagAccept = 0u;
constexpr uint32_t kTagRace = 1u;

// Accept uniform of draft position `pos` of global request `req`: the top 52
// bits m of words 0..1 give u = (2m + 1) 2^-53, exact and strictly inside
// (0, 1) as a double (velog "vLLM 커널은 이 규칙을 어떻게 옮겼나": float64
// uniforms, so u = 0 never lets a p = 0 token through).
__device__ __forceinline__ double accept_uniform(unsigned long long seed, long long req,
                                                 int pos) {
  const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)req, kTagAccept),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  const unsigned long long bits = ((unsigned long long)w.x << 32) | w.y;
  const unsigned long long m52 = bits >> 12;
  return (double)(2ull * m52 + 1ull) * 0x1p-53;
}

// Race uniform from one Philox word: U = (2 (w >> 9) + 1) 2^-24, exact in
// float and strictly inside (0, 1), so E = -ln U is finite and positive.
__device__ __forceinline__ float race_uniform_from_word(uint32_t w) {
  return (float)(2u * (w >> 9) + 1u) * 0x1p-24f;
}

// The four race words of vocabulary group g (entries 4g .. 4g+3) of the row
// at position `pos` of global request `req`.
__device__ __forceinline__ uint4 race_words(unsigned long long seed, long long req, int pos,
                                            uint32_t g) {
  return philox4x32_10(make_uint4(g, (uint32_t)pos, (uint32_t)req, kTagRace),
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}

}  // namespace sv
