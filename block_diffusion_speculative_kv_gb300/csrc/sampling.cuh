// Temperature sampling of drafted tokens by the Gumbel-max rule.
//
// "DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.4:
// at temperature 0 a block position drafts the argmax of its logits, at
// temperature T > 0 a sample from softmax(logits / T).  The sample is the
// token maximising the score s_v = l_v / T + G_v, G_v = -log(-log U_v) with
// U_v uniform on (0, 1).  Taking the K best scores instead of the best one
// draws K tokens without replacement (the Gumbel-top-k property).
//
// U_v comes from the counter-based SplitMix64 generator (Steele, Lea and
// Flood, "Fast splittable pseudorandom number generators", 2014): output k of
// the generator seeded with `seed` mixes seed + k * golden-gamma.  Element v of
// counter row r uses k = (r << 32 | v) + 1; U = (top 23 bits + 1/2) / 2^23 is
// exact in fp32 and strictly inside (0, 1).  The score is rounded like the
// plain fp32 expression l * (1/T) + G: a multiply and an add, never fused.
#pragma once

#include <cstdint>

namespace dfl {

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t k) {
  uint64_t z = seed + k * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// G for element v of counter row `row`.
__device__ __forceinline__ float gumbel_noise(uint64_t seed, long long row, int v) {
  const uint64_t k = (((uint64_t)row << 32) | (uint32_t)v) + 1ull;
  const uint32_t top = (uint32_t)(splitmix64(seed, k) >> 41);
  const float u = __uint2float_rn(2u * top + 1u) * 5.9604644775390625e-8f;  // 2^-24
  return -logf(-logf(u));
}

__device__ __forceinline__ float gumbel_score(float logit, float inv_t, uint64_t seed,
                                              long long row, int v) {
  return __fadd_rn(__fmul_rn(logit, inv_t), gumbel_noise(seed, row, v));
}

// log q of a sampled token recovered from its score: (s - G) * T - lse.
__device__ __forceinline__ float sampled_logq(float score, float t, uint64_t seed, long long row,
                                              int v, float lse) {
  return (score - gumbel_noise(seed, row, v)) * t - lse;
}

}  // namespace dfl
