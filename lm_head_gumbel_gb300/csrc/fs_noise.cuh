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

// Hardware base-2 logarithm (flush-to-zero form: every argument used here is
// a normal number, so no subnormal handling is needed).
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2Ln2 = -0.5287663729448977f;  // log2(ln 2)

// The Gumbel noise of one random word, in base-2 units: returns
// q = log2(-log2 u), so that g = -log(-log u) = -ln2 * (q + log2(ln 2)).
//
// u = ((w & 0x7fffff) + 1/2) 2^-23: built from the bit pattern 1 + k 2^-23
// minus (1 - 2^-24), exact (at most 24 significant bits), so 0 < u < 1;
// x = 1 - u is exact as well.  Then E = -log2 u:
//  - E decides the largest noise values (u near 1, E tiny), which are the ones
//    that win the argmax, so there it must be accurate relative to E.  For
//    x < 2^-5 it uses the Taylor series -log2(1 - x) = log2(e) (x + x^2/2 +
//    x^3/3 + x^4/4 + x^5/5 + ...), truncated after x^5/5 (relative truncation
//    error below x^5/6 < 6e-9); otherwise the hardware log2 of u, whose
//    absolute error (< 2^-22 on [1/2, 2]) is then at most ~5e-6 relative to
//    |log2 u| >= 0.046;
//  - q = log2 E only needs absolute accuracy.
// The resulting g differs from the exact fp64 -log(-log u) by a few 1e-6.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
  const float f = __uint_as_float(0x3F800000u | (w & 0x7FFFFFu));  // 1 + k 2^-23
  return f - 0x1.fffffep-1f;                                        // k 2^-23 + 2^-24
}

__device__ __forceinline__ float gumbel_log2_from_word(uint32_t w) {
  const float u = uniform_from_word(w);
  const float x = 1.0f - u;
  float ser = fmaf(x, 0.2f * kLog2e, 0.25f * kLog2e);
  ser = fmaf(x, ser, kLog2e / 3.0f);
  ser = fmaf(x, ser, 0.5f * kLog2e);
  ser = fmaf(x, ser, kLog2e);
  const float E = (x < 0x1p-5f) ? x * ser : -lg2_approx(u);
  return lg2_approx(E);
}

// Gumbel(0,1) noise of one random word, in natural units.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  return -kLn2 * (gumbel_log2_from_word(w) + kLog2Ln2);
}

__device__ __forceinline__ uint32_t select_word(uint4 r, uint32_t which) {
  return which == 0 ? r.x : which == 1 ? r.y : which == 2 ? r.z : r.w;
}

}  // namespace fs
