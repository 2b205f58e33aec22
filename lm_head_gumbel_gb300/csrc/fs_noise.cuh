// fs_noise.cuh -- counter-based Gumbel noise for the sampling epilogue.
//
// g = -log(-log u) (aitrends.kr write-up on FlashSampling, "Stage 1 (Fused
// Kernel)"), generated in fp32 as the write-up's implementation notes state.
// The uniform u comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): ten rounds of two
// 32x32->64-bit multiplies whose halves are xored with the other counter words
// and the round key, the key advancing by the Weyl increments between rounds.
//
// Element (b, v) of a call with (seed_b, offset) uses
//   key     = (seed_b low word, seed_b high word)
//   counter = (v >> 2, b, offset low word, offset high word)
// and output word v & 3, so one Philox evaluation serves four consecutive
// vocabulary ids of a row.
#pragma once

#include <cstdint>

namespace fs {

struct PhiloxKey {
  uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 x, PhiloxKey key) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kMul0, x.x), lo0 = kMul0 * x.x;
    const uint32_t hi1 = __umulhi(kMul1, x.z), lo1 = kMul1 * x.z;
    x = make_uint4(hi1 ^ x.y ^ k0, lo1, hi0 ^ x.w ^ k1, lo0);
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  return x;
}

// Uniform in (0,1) from the top 23 bits of a word: ((w >> 9) + 1/2) * 2^-23.
// Every value is exact in fp32 (at most 24 significant bits), so u is never
// 0 or 1 and log(u) is finite and nonzero.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
  return fmaf(static_cast<float>(w >> 9), 0x1p-23f, 0x1p-24f);
}

// Gumbel(0,1) by inversion.  The inner log must be accurate relative to its
// (tiny) result when u is close to 1 -- those are the largest noise values,
// the ones that win the argmax -- so both logs use the IEEE-accurate logf.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  const float u = uniform_from_word(w);
  return -logf(-logf(u));
}

__device__ __forceinline__ uint32_t select_word(uint4 r, uint32_t which) {
  return which == 0 ? r.x : which == 1 ? r.y : which == 2 ? r.z : r.w;
}

}  // namespace fs
