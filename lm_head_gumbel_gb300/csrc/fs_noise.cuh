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

constexpr uint32_t kPhiloxMul0 = 0xD2511F53u, kPhiloxMul1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxWeyl0 = 0x9E3779B9u, kPhiloxWeyl1 = 0xBB67AE85u;

// The ten round keys of one 64-bit seed, computed once per row.
struct PhiloxSchedule {
  uint32_t k0[10], k1[10];
  __device__ __forceinline__ explicit PhiloxSchedule(uint64_t seed) {
    uint32_t a = static_cast<uint32_t>(seed), b = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      k0[r] = a;
      k1[r] = b;
      a += kPhiloxWeyl0;
      b += kPhiloxWeyl1;
    }
  }
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 x, const PhiloxSchedule& ks) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxMul0) * x.x;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxMul1) * x.z;
    x = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ x.y ^ ks.k0[r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ x.w ^ ks.k1[r], static_cast<uint32_t>(p0));
  }
  return x;
}

// Gumbel(0,1) noise from one random word, in fp32.
//
// u = ((w >> 9) + 1/2) 2^-23: built from the bit pattern 1 + k 2^-23 minus
// (1 - 2^-24), exact (at most 24 significant bits), so 0 < u < 1; x = 1 - u is
// exact as well.  Then g = -ln(e) with e = -ln(u):
//  - the inner log decides the largest noise values (u near 1, e tiny), which
//    are the ones that win the argmax, so there it must be accurate relative to
//    e.  For x < 2^-5 it uses the Taylor series of -ln(1 - x) = x (1 + x/2 +
//    x^2/3 + x^3/4 + x^4/5 + ...), truncated after x^4/5 (relative truncation
//    error below x^5/6 < 6e-9); otherwise -ln2 * log2(u) with the hardware base-2
//    logarithm, whose absolute error (< 2^-22 on [1/2, 2]) is then at most
//    ~5e-6 relative to |log2 u| >= 0.046;
//  - the outer log only needs absolute accuracy: -ln2 * log2(e).
// The noise differs from the exact fp64 -log(-log u) by a few 1e-6 at most.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  constexpr float kLn2 = 0.693147180559945f;
  const float f = __uint_as_float(0x3F800000u | (w >> 9));  // 1 + k 2^-23
  const float u = f - 0x1.fffffep-1f;                        // k 2^-23 + 2^-24
  const float x = 1.0f - u;
  float ser = fmaf(x, 0.2f, 0.25f);
  ser = fmaf(x, ser, 0.333333343f);
  ser = fmaf(x, ser, 0.5f);
  ser = fmaf(x, ser, 1.0f);
  const float e = (x < 0x1p-5f) ? x * ser : -kLn2 * __log2f(u);
  return -kLn2 * __log2f(e);
}

__device__ __forceinline__ uint32_t select_word(uint4 r, uint32_t which) {
  return which == 0 ? r.x : which == 1 ? r.y : which == 2 ? r.z : r.w;
}

}  // namespace fs
