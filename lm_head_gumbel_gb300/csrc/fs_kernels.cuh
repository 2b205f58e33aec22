// fs_kernels.cuh -- the device code of fused LM-head + exact Gumbel-max sampling
// on GB300 (sm_103a).  Included by fs_sample.cu only (it defines device
// variables); the host side (argument checks, tensor maps, launches, the C ABI)
// is there.
//
// Stage 1 (the aitrends.kr write-up on FlashSampling, "Stage 1 (Fused
// Kernel)"; tomesphere abstract, "compute logits tile-by-tile on chip, add
// Gumbel noise, keep only one maximizer per row and per vocabulary tile"):
// a persistent, warp-specialised kernel.  For up to 128 rows (and odd numbers
// of 128-row blocks) each work unit is a 128-row batch block x 256-id
// vocabulary block of the logits l = H W^T, computed by one CTA; for an even
// number of batch blocks, CTA pairs compute 256 x 256 units with cta_group::2
// MMAs (stage1_pair_kernel below).  Single-CTA roles:
//   warp 0    TMA producer (one elected lane issues): streams 64-wide K
//             slices of W (256 x 64) and H (up to 128 x 64) into a shared-
//             memory ring of 4-5 stages (128-byte swizzle; the fewer H rows,
//             the more stages)
//   warp 1    tcgen05 MMA issuer (one elected lane issues): M=128, N=256,
//             K=16 bf16 MMAs accumulate the unit's logits in tensor memory
//             (fp32, 256 columns); two accumulators so the epilogue of one
//             unit overlaps the MMAs of the next
//   warps 2-9 epilogue: each thread owns one batch row and 128 vocabulary
//             columns (one output tile); it reads its logits from tensor
//             memory, scales by 1/T, masks, adds Philox Gumbel noise, and
//             keeps the running (max, argmax) and optionally the log-sum-exp
//             -- or, in the top-K modes, the best 4 or 16 (score, id).  For a
//             CTA's last unit the noise is made while its W streams in and
//             parked in the idle accumulator (noise_ahead), since nothing
//             overlaps that unit's epilogue
// Only (m_t, i_t[, L_t]) -- or the top-K list -- per (row, 128-id tile)
// leaves the chip.
//
// Stage 2 ("Stage 2 (Reduction)") is fused: each tile winner is folded into a
// per-row 64-bit key with an order-free atomic max, and the last CTA to finish
// writes the sampled ids (lowest id on ties) and clears the keys.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "fs_noise.cuh"
#include "fs_ptx.cuh"
#include "fs_sample.h"

namespace fs {

constexpr int kBlockM = 128;   // batch rows per unit = tensor-memory lanes
constexpr int kBlockN = 256;   // vocabulary ids per unit = accumulator columns
constexpr int kBlockK = 64;    // bf16 elements per 128-byte swizzled row
constexpr int kUmmaK = 16;     // K of one kind::f16 MMA
constexpr int kMaxStages = 5;  // ring depth: as many stages as fit kRingBytes, at most 5
constexpr int kTileV = FS_TILE;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kSmemA = kBlockM * kBlockK * 2;  // H slice of 128 rows, 16 KB
constexpr uint32_t kSmemB = kBlockN * kBlockK * 2;  // W slice, 32 KB
constexpr uint32_t kRingBytes = 200 * 1024;         // stages of H rows + W slice
constexpr uint32_t kTmemCols = 2 * kBlockN;         // two fp32 accumulators
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBlockM, kBlockN);
constexpr size_t kBarOffset = kRingBytes;
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kBarOffset + 256;
static_assert(kBlockN == 2 * kTileV, "one unit covers two output tiles");
static_assert(kBlockK * 2 == 128, "one K slice row is one 128-byte swizzle row");

enum : int { kErrWaitTimeout = 1 };

__device__ int g_error_word = 0;

struct Stage1Params {
  int32_t B, V;
  int32_t n_tiles;   // ceil(V / 128)
  int32_t n_mt;      // ceil(B / 128)
  int32_t n_kb;      // ceil(d / 64)
  const float* temperature;
  const uint32_t* mask;
  int64_t mask_ld;
  const uint64_t* seeds;
  uint64_t seed, offset;
  float* tile_max;             // per-tile outputs, or null
  int32_t* tile_idx;
  float* tile_lse;
  int64_t* out_idx;            // sampled ids, or null (per-tile outputs only)
  int64_t* out_idx_host;       // optional second copy of the ids in mapped host memory
  float* out_max;              // optional: the row's largest noisy score
  int32_t vocab_offset;        // global id of W's first row (a multiple of 4)
  unsigned long long* row_keys;  // [B] packed (score, id) maxima, zero between calls
  uint32_t* ticket;            // CTAs finished so far, wraps back to zero
  float* topk_score;           // top-K modes: [B, n_tiles, cap] best scores per tile
  int32_t* topk_idx;           //              [B, n_tiles, cap] their global ids
  uint64_t wait_limit_ns;
  uint32_t h_box_rows;  // rows of the H box: min(128, B rounded up to 8)
  // Single-CTA ring: a stage is the H box (h_box_rows x 128 bytes, whole
  // 1 KB swizzle atoms) followed by the W slice; small batches get more
  // stages, so more of W is in flight.
  uint32_t n_stages;
  uint32_t stage_bytes;
  // Launched to overlap the kernel that writes H and the per-row inputs
  // (programmatic dependent launch): W streams at once, H and the per-row
  // inputs are read only after the grid dependency is resolved.
  uint32_t pdl;
  // CTA-pair kernel with more than one pair batch block: groups of pairs
  // walking the same vocabulary blocks (pair_unit); 0 for the plain order.
  int32_t pair_groups;        // groups of n_mp pairs
  int32_t pair_group_blocks;  // vocabulary blocks each group walks
};

// The producer's H copies of the first ring fill, held back until the grid
// dependency is resolved when the kernel overlaps the one writing H.
struct DeferredH {
  int n = 0;
  uint32_t stage[8];
  int kb[8], row[8];
};
static_assert(kMaxStages <= 8, "a ring fill of deferred H copies fits DeferredH");

// Bounded mbarrier waits: past the limit the CTA raises its abort flag and
// the device error word, and every role winds down instead of spinning.
struct Waiter {
  volatile uint32_t* abort_flag;
  uint64_t limit_ns;

  __device__ bool wait(uint64_t* bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    while (true) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if (*abort_flag) return false;
      if (ptx::global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1u;
        atomicOr(&g_error_word, kErrWaitTimeout);
        return false;
      }
    }
  }
  // The same wait for a warp whose lanes all poll the barrier: every lane
  // gets the same answer (a lane that gave up makes the whole warp give up).
  __device__ bool wait_warp(uint64_t* bar, uint32_t parity) const {
    return __all_sync(0xFFFFFFFFu, wait(bar, parity));
  }
  // Used while winding down: ignores the abort flag, still bounded.
  __device__ bool drain(uint64_t* bar, uint32_t parity) const {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (ptx::global_timer_ns() - t0 > limit_ns) {
        atomicOr(&g_error_word, kErrWaitTimeout);
        return false;
      }
    }
    return true;
  }
};

// (score, id) as one unsigned 64-bit key whose order is: higher score first,
// then lower id (the tie rule).  The score's bits are mapped to an order-
// preserving unsigned word (-0 folded into +0); every valid key is nonzero.
__device__ __forceinline__ unsigned long long pack_key(float m, int32_t idx) {
  uint32_t b = __float_as_uint(m + 0.0f);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ int64_t unpack_idx(unsigned long long key) {
  return key == 0ull ? int64_t(-1) : int64_t(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ float unpack_score(unsigned long long key) {
  if (key == 0ull) return -INFINITY;
  const uint32_t b = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b);
}

// One 32-column chunk of a sampling row, in base-2 units: s2 = l * (log2 e / T)
// - log2(-log2 u), which is s * log2(e) shifted by a constant, so it has the
// same argmax.  Updates the running maximum `best2` and, if this chunk holds
// a new maximum, its position `best_j` in the chunk (else leaves -1).
template <bool kMasked>
__device__ __forceinline__ void sample_chunk(const uint32_t (&r)[32], uint32_t allow,
                                             float scale2, uint32_t ctr0, uint32_t ctr_row,
                                             uint32_t ctr_lo, uint32_t ctr_hi,
                                             const PhiloxSchedule& ks, float& best2,
                                             int& best_j) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint4 rnd = philox4x32_10(make_uint4(ctr0 + g, ctr_row, ctr_lo, ctr_hi), ks);
    const uint32_t words[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = g * 4 + i;
      const float s2 = fmaf(__uint_as_float(r[j]), scale2, -gumbel_log2_from_word(words[i]));
      if ((!kMasked || ((allow >> j) & 1u)) && s2 > best2) {
        best2 = s2;
        best_j = j;
      }
    }
  }
}

template <bool kMasked>
__device__ __forceinline__ void greedy_chunk(const uint32_t (&r)[32], uint32_t allow,
                                             float& best, int& best_j) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float l = __uint_as_float(r[j]);
    if ((!kMasked || ((allow >> j) & 1u)) && l > best) {
      best = l;
      best_j = j;
    }
  }
}

// sample_chunk with the chunk's noise q = log2(-log2 u) already made
// (noise_ahead): the same sums in the same order, so the same result.
template <bool kMasked>
__device__ __forceinline__ void sample_chunk_pre(const uint32_t (&r)[32], const uint32_t (&q)[32],
                                                 uint32_t allow, float scale2, float& best2,
                                                 int& best_j) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float s2 = fmaf(__uint_as_float(r[j]), scale2, -__uint_as_float(q[j]));
    if ((!kMasked || ((allow >> j) & 1u)) && s2 > best2) {
      best2 = s2;
      best_j = j;
    }
  }
}

// The noise of a CTA's last unit, made before its logits exist.  Nothing
// overlaps the epilogue of a CTA's last unit, but the noise does not depend on
// the logits: while the unit's W slices stream in, each epilogue warp (idle
// once the unit before is done) writes q = log2(-log2 u) for its 32 rows and
// 128 ids into its own lanes and columns of the other accumulator buffer,
// which no MMA writes any more.  The last epilogue then reads it beside the
// logits.  A warp whose rows are all greedy or past the batch writes nothing.
__device__ __forceinline__ void noise_ahead(const Stage1Params& p, uint32_t ntaddr, int row,
                                            int tile) {
  const bool valid_row = row < p.B;
  float T = 1.0f;
  uint64_t seed = p.seed;
  if (valid_row) {
    if (p.temperature) T = p.temperature[row];
    if (p.seeds) seed = p.seeds[row];
  }
  const bool sampled = valid_row && T > 0.0f && !isinf(T);
  if (!__any_sync(0xFFFFFFFFu, sampled)) return;
  // Every lane makes noise (the unused lanes' too), so the warp stays converged.
  const PhiloxSchedule ks(seed);
  const uint32_t ctr_row = static_cast<uint32_t>(row);
  const uint32_t ctr_lo = static_cast<uint32_t>(p.offset);
  const uint32_t ctr_hi = static_cast<uint32_t>(p.offset >> 32);
#pragma unroll 1
  for (int c = 0; c < kTileV / 32; ++c) {
    const uint32_t ctr0 = static_cast<uint32_t>((p.vocab_offset + tile * kTileV + c * 32) >> 2);
    uint32_t q[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint4 rnd = philox4x32_10(make_uint4(ctr0 + g, ctr_row, ctr_lo, ctr_hi), ks);
      q[4 * g + 0] = __float_as_uint(gumbel_log2_from_word(rnd.x));
      q[4 * g + 1] = __float_as_uint(gumbel_log2_from_word(rnd.y));
      q[4 * g + 2] = __float_as_uint(gumbel_log2_from_word(rnd.z));
      q[4 * g + 3] = __float_as_uint(gumbel_log2_from_word(rnd.w));
    }
    ptx::tmem_st_32x32b_x32(ntaddr + uint32_t(c * 32), q);
  }
  ptx::tmem_wait_st();
}

// The allow-words of one row's 128-id tile, all loaded before the tile's
// chunks are processed (a word loaded inside the chunk loop would be waited
// for after each chunk's tensor-memory load).  Only words holding ids below V
// are read -- the ceil(V/32) words a mask row has -- and ids at or past V are
// allowed nowhere.
struct TileMask {
  uint32_t w[kTileV / 32];
  __device__ __forceinline__ TileMask(const uint32_t* mrow, int v_tile, int V) {
#pragma unroll
    for (int c = 0; c < kTileV / 32; ++c) {
      const int v0 = v_tile + c * 32;
      const int n_in = V - v0;
      w[c] = n_in <= 0 ? 0u : (mrow != nullptr ? mrow[v0 >> 5] : 0xFFFFFFFFu);
      if (n_in > 0 && n_in < 32) w[c] &= (1u << n_in) - 1u;
    }
  }
  // Word c, for a chunk index known only at run time, without local memory.
  __device__ __forceinline__ uint32_t at(int c) const {
    return c == 0 ? w[0] : c == 1 ? w[1] : c == 2 ? w[2] : w[3];
  }
};
static_assert(kTileV / 32 == 4, "TileMask::at picks one of four words");

// One thread, one batch row, one 128-id output tile: read the logits from
// tensor memory 32 columns at a time and reduce them to (m_t, i_t[, L_t]).
// With kPreNoise the noise is read from tensor memory at ntaddr (noise_ahead)
// instead of being made here.
template <bool kWantLse, bool kPreNoise>
__device__ __forceinline__ void epilogue_tile(const Stage1Params& p, uint32_t taddr, int row,
                                              int tile, uint32_t ntaddr) {
  const bool valid_row = row < p.B;
  float T = 1.0f;
  uint64_t seed = p.seed;
  const uint32_t* mrow = nullptr;
  if (valid_row) {
    if (p.temperature) T = p.temperature[row];
    if (p.seeds) seed = p.seeds[row];
    if (p.mask) mrow = p.mask + int64_t(row) * p.mask_ld;
  }
  const bool greedy = !(T > 0.0f) || isinf(T);
  const float scale2 = greedy ? 1.0f : kLog2e / T;  // l -> l' in base-2 units
  const PhiloxSchedule ks(seed);
  const uint32_t ctr_row = static_cast<uint32_t>(row);
  const uint32_t ctr_lo = static_cast<uint32_t>(p.offset);
  const uint32_t ctr_hi = static_cast<uint32_t>(p.offset >> 32);
  // noise_ahead wrote noise only for warps with a sampled row.
  const bool load_noise = kPreNoise && __any_sync(0xFFFFFFFFu, valid_row && !greedy);

  float best = -INFINITY;  // greedy: max l; sampling: max s2
  int32_t best_idx = -1;
  float run_max = -INFINITY, run_sum = 0.0f;  // base-2 log-sum-exp state
  const int v_tile = tile * kTileV;
  const TileMask tm(mrow, v_tile, p.V);  // mrow is null for rows past the batch

#pragma unroll 1
  for (int c = 0; c < kTileV / 32; ++c) {
    uint32_t r[32];
    uint32_t qn[32];
    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * 32), r);
    if (load_noise) ptx::tmem_ld_32x32b_x32(ntaddr + uint32_t(c * 32), qn);
    ptx::tmem_wait_ld();
    const int v0 = v_tile + c * 32;
    const uint32_t allow = valid_row ? tm.at(c) : 0xFFFFFFFFu;
    // The mask test is skipped only when no lane of the warp needs it: a
    // per-lane choice would run both forms one after the other.
    const bool unmasked = __all_sync(0xFFFFFFFFu, allow == 0xFFFFFFFFu);
    if (!valid_row) continue;
    int best_j = -1;
    if (greedy) {
      if (unmasked)
        greedy_chunk<false>(r, allow, best, best_j);
      else
        greedy_chunk<true>(r, allow, best, best_j);
    } else if (kPreNoise) {
      if (unmasked)
        sample_chunk_pre<false>(r, qn, allow, scale2, best, best_j);
      else
        sample_chunk_pre<true>(r, qn, allow, scale2, best, best_j);
    } else {
      const uint32_t ctr0 = static_cast<uint32_t>((p.vocab_offset + v0) >> 2);
      if (unmasked)
        sample_chunk<false>(r, allow, scale2, ctr0, ctr_row, ctr_lo, ctr_hi, ks, best, best_j);
      else
        sample_chunk<true>(r, allow, scale2, ctr0, ctr_row, ctr_lo, ctr_hi, ks, best, best_j);
    }
    if (best_j >= 0) best_idx = p.vocab_offset + v0 + best_j;
    if (kWantLse && !greedy) {
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if ((allow >> j) & 1u) cm = fmaxf(cm, __uint_as_float(r[j]) * scale2);
      if (cm > -INFINITY) {
        const float m_new = fmaxf(run_max, cm);
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((allow >> j) & 1u) acc += ex2_approx(fmaf(__uint_as_float(r[j]), scale2, -m_new));
        run_sum = fmaf(run_sum, ex2_approx(run_max - m_new), acc);
        run_max = m_new;
      }
    }
  }
  if (!valid_row) return;
  // Back to natural units: s = ln2 * (s2 - log2(ln 2)).
  const float m = (greedy || best_idx < 0) ? best : kLn2 * (best - kLog2Ln2);
  // Fold the tile's winner into the row's running maximum: the key orders by
  // score, then by lower id, so the result does not depend on arrival order.
  if (p.out_idx != nullptr && best_idx >= 0) atomicMax(p.row_keys + row, pack_key(m, best_idx));
  if (p.tile_max == nullptr) return;
  const int64_t o = int64_t(row) * p.n_tiles + tile;
  p.tile_max[o] = m;
  p.tile_idx[o] = best_idx;
  if (kWantLse) {
    float L = best;  // greedy rows: the largest unmasked logit
    if (!greedy) L = run_max > -INFINITY ? (run_max + lg2_approx(run_sum)) * kLn2 : -INFINITY;
    p.tile_lse[o] = L;
  }
}

// Insert (s, id) into a list sorted by decreasing score whose last entry it
// beats.  Equal scores keep their order, so with ids visited in increasing
// order the lower id stays first (the tie rule).
template <int KC>
__device__ __forceinline__ void topk_insert(float (&ts)[KC], int32_t (&ti)[KC], float s,
                                            int32_t id) {
  ts[KC - 1] = s;
  ti[KC - 1] = id;
#pragma unroll
  for (int q = KC - 1; q > 0; --q) {
    const bool up = ts[q] > ts[q - 1];
    const float a = ts[q], b = ts[q - 1];
    const int32_t ia = ti[q], ib = ti[q - 1];
    ts[q - 1] = up ? a : b;
    ts[q] = up ? b : a;
    ti[q - 1] = up ? ia : ib;
    ti[q] = up ? ib : ia;
  }
}

// v[j] for a lane-varying j, without local memory: a 5-level select tree.
__device__ __forceinline__ float select32(const float (&v)[32], uint32_t j) {
  float a[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) a[q] = (j & 16u) ? v[q + 16] : v[q];
#pragma unroll
  for (int q = 0; q < 8; ++q) a[q] = (j & 8u) ? a[q + 8] : a[q];
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q] = (j & 4u) ? a[q + 4] : a[q];
#pragma unroll
  for (int q = 0; q < 2; ++q) a[q] = (j & 2u) ? a[q + 2] : a[q];
  return (j & 1u) ? a[1] : a[0];
}

// A thread's running top-KC list for the row it is working on, across the
// tiles of consecutive units with that row (a "stretch"); sorted best first,
// in base-2 units for sampled rows.
template <int KC>
struct TopKState {
  float s[KC];
  int32_t i[KC];
  int row = -1;        // the stretch's row, -1 before the first tile
  int last_tile = -1;  // the slot the list is written to
  bool greedy = false;
};

// Write the stretch's list to the workspace slot of its last tile (the
// stretch's other tiles hold an empty list), in natural units.
template <int KC>
__device__ __forceinline__ void topk_flush(const Stage1Params& p, const TopKState<KC>& st) {
  if (st.row < 0) return;
  const int64_t o = (int64_t(st.row) * p.n_tiles + st.last_tile) * KC;
  // The slot is KC contiguous scores then (elsewhere) KC ids, 16-byte aligned.
  float4* s4 = reinterpret_cast<float4*>(p.topk_score + o);
  int4* i4 = reinterpret_cast<int4*>(p.topk_idx + o);
#pragma unroll
  for (int q = 0; q < KC; q += 4) {
    float m[4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
      m[x] = (st.greedy || st.i[q + x] < 0) ? st.s[q + x] : kLn2 * (st.s[q + x] - kLog2Ln2);
    s4[q / 4] = make_float4(m[0], m[1], m[2], m[3]);
    i4[q / 4] = make_int4(st.i[q], st.i[q + 1], st.i[q + 2], st.i[q + 3]);
  }
}

// Top-K form of epilogue_tile.  By the Gumbel-top-k property the K largest
// noisy scores of a row are K draws without replacement from softmax(l'), in
// draw order.  Each thread keeps the KC best (score, id) of everything it has
// seen of its row; an element enters only if it beats the list's last entry,
// which is safe because an element of the row's K <= KC best is among the KC
// best of any subset holding it.  Per 32-id chunk every lane marks its
// entering candidates, then the warp runs as many insertion rounds as the
// lane with most candidates needs (one candidate per lane and round, lowest
// id first, so ties keep the lower id), instead of one warp-wide insertion
// per id that any lane wants.
template <int KC>
__device__ __forceinline__ void epilogue_tile_topk(const Stage1Params& p, uint32_t taddr,
                                                   int row, int tile, TopKState<KC>& st,
                                                   uint32_t ntaddr, bool pre) {
  const bool valid_row = row < p.B;
  float T = 1.0f;
  uint64_t seed = p.seed;
  const uint32_t* mrow = nullptr;
  if (valid_row) {
    if (p.temperature) T = p.temperature[row];
    if (p.seeds) seed = p.seeds[row];
    if (p.mask) mrow = p.mask + int64_t(row) * p.mask_ld;
    if (st.row != row) {  // a new stretch
      topk_flush<KC>(p, st);
#pragma unroll
      for (int q = 0; q < KC; ++q) {
        st.s[q] = -INFINITY;
        st.i[q] = -1;
      }
      st.row = row;
    }
    // The slot is empty unless the stretch's list lands here.  Its first id
    // alone marks it, but written as whole 32-byte sectors (16 bytes at
    // KC = 4, whose neighbour tile writes the other half at about the same
    // time): a partly written sector is read back from DRAM when it leaves
    // the L2, beside the W stream.
    int4* m4 = reinterpret_cast<int4*>(p.topk_idx + (int64_t(row) * p.n_tiles + tile) * KC);
    m4[0] = make_int4(-1, -1, -1, -1);
    if (KC >= 8) m4[1] = make_int4(-1, -1, -1, -1);
    st.last_tile = tile;
  }
  const bool greedy = !(T > 0.0f) || isinf(T);
  st.greedy = greedy;
  const float scale2 = greedy ? 1.0f : kLog2e / T;
  const PhiloxSchedule ks(seed);
  const uint32_t ctr_row = static_cast<uint32_t>(row);
  const uint32_t ctr_lo = static_cast<uint32_t>(p.offset);
  const uint32_t ctr_hi = static_cast<uint32_t>(p.offset >> 32);
  // noise_ahead wrote noise only for warps with a sampled row.
  const bool load_noise = pre && __any_sync(0xFFFFFFFFu, valid_row && !greedy);
  const int v_tile = tile * kTileV;
  const TileMask tm(mrow, v_tile, p.V);  // mrow is null for rows past the batch
#pragma unroll 1
  for (int c = 0; c < kTileV / 32; ++c) {
    uint32_t r[32];
    float sc[32];
    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * 32), r);
    if (load_noise)  // the noise lands in sc; the scores are made in place below
      ptx::tmem_ld_32x32b_x32(ntaddr + uint32_t(c * 32), reinterpret_cast<uint32_t(&)[32]>(sc));
    ptx::tmem_wait_ld();
    const int v0 = v_tile + c * 32;
    const int32_t id0 = p.vocab_offset + v0;
    uint32_t cand = 0u;
    if (valid_row) {
      const uint32_t allow = tm.at(c);
      if (greedy) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sc[j] = __uint_as_float(r[j]);
      } else if (pre) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sc[j] = fmaf(__uint_as_float(r[j]), scale2, -sc[j]);
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 rnd = philox4x32_10(
              make_uint4(static_cast<uint32_t>(id0 >> 2) + g, ctr_row, ctr_lo, ctr_hi), ks);
          const uint32_t words[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sc[g * 4 + q] =
                fmaf(__uint_as_float(r[g * 4 + q]), scale2, -gumbel_log2_from_word(words[q]));
        }
      }
      const float tau = st.s[KC - 1];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        cand |= (((allow >> j) & 1u) && sc[j] > tau) ? (1u << j) : 0u;
    }
    while (__any_sync(0xFFFFFFFFu, cand != 0u)) {
      if (cand != 0u) {
        const uint32_t j = uint32_t(__ffs(cand) - 1);
        cand &= cand - 1u;
        const float v = select32(sc, j);
        if (v > st.s[KC - 1]) topk_insert<KC>(st.s, st.i, v, id0 + int32_t(j));
      }
    }
  }
}

// Stage 2 ("Stage 2 (Reduction)"), fused: the last CTA to finish turns the
// per-row maxima into sampled ids and clears them for the next call.  The
// ticket wraps to zero on the last arrival, so it too is left cleared.  Called
// by every thread of every CTA once its work is done (and its row-key updates
// fenced).
__device__ __forceinline__ void finish_rows(const Stage1Params& p) {
  if (p.out_idx == nullptr) return;
  __shared__ uint32_t s_is_last;
  if (threadIdx.x == 0) {
    __threadfence();
    s_is_last = (atomicInc(p.ticket, gridDim.x - 1u) == gridDim.x - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (s_is_last) {
    __threadfence();
    for (int r = threadIdx.x; r < p.B; r += blockDim.x) {
      const unsigned long long key = atomicExch(p.row_keys + r, 0ull);
      const int64_t id = unpack_idx(key);
      p.out_idx[r] = id;
      if (p.out_idx_host != nullptr) p.out_idx_host[r] = id;
      if (p.out_max != nullptr) p.out_max[r] = unpack_score(key);
    }
  }
}

// Epilogue modes (a template parameter of both stage-1 kernels).
enum : int {
  kModeSample = 0,  // (m_t, i_t) per tile, row maxima
  kModeLse = 1,     // ... plus the tile log-sum-exp
  kModeTop4 = 2,    // the 4 best (score, id) per tile, for K <= 4 draws without replacement
  kModeTop16 = 3,   // the 16 best, for K <= 16
};
__host__ __device__ constexpr int topk_cap(int mode) {
  return mode == kModeTop4 ? 4 : mode == kModeTop16 ? 16 : 1;
}
template <int kMode>
constexpr bool kTopkMode = kMode == kModeTop4 || kMode == kModeTop16;

// Per-thread epilogue state carried across units: the running top-K list in
// the top-K modes, nothing otherwise.
struct NoState {};
template <int kMode>
using EpilogueState =
    typename std::conditional<(kMode == kModeTop4 || kMode == kModeTop16),
                              TopKState<topk_cap(kMode)>, NoState>::type;

// One unit's epilogue for one thread.  With `pre` the noise is read from
// tensor memory at ntaddr (noise_ahead) instead of being made.  The sampling
// modes inline a form of each; the top-K modes test the flag inside one form
// (two inlined forms beside the lists needed more registers than a thread
// has, and spilled).
template <int kMode>
__device__ __forceinline__ void epilogue_unit(const Stage1Params& p, uint32_t taddr, int row,
                                              int tile, EpilogueState<kMode>& st,
                                              uint32_t ntaddr, bool pre) {
  if constexpr (kMode == kModeSample || kMode == kModeLse) {
    if (pre)
      epilogue_tile<kMode == kModeLse, true>(p, taddr, row, tile, ntaddr);
    else
      epilogue_tile<kMode == kModeLse, false>(p, taddr, row, tile, 0u);
  } else {
    epilogue_tile_topk<topk_cap(kMode)>(p, taddr, row, tile, st, ntaddr, pre);
  }
}

// After a thread's last unit: the top-K modes write the open stretch's list.
template <int kMode>
__device__ __forceinline__ void epilogue_finish(const Stage1Params& p, EpilogueState<kMode>& st) {
  if constexpr (kMode == kModeTop4 || kMode == kModeTop16) topk_flush<topk_cap(kMode)>(p, st);
}

// Single-CTA stage 1: a unit is (vocabulary block vt of 256 ids, batch block mt
// of 128 rows), computed by one CTA with M = 128, N = 256 MMAs; units are
// ordered vocabulary-major so the batch blocks of one vocabulary block run on
// neighbouring CTAs at the same time and the second read of W hits L2.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_kernel(const __grid_constant__ CUtensorMap tmap_h,
                  const __grid_constant__ CUtensorMap tmap_w, const Stage1Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty_bar = full_bar + kMaxStages;
  uint64_t* tfull_bar = empty_bar + kMaxStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Vocabulary blocks from the tile count: V + 255 overflows 32 bits near V = 2^31.
  const int n_units = ((p.n_tiles + 1) / 2) * p.n_mt;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.n_stages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull_bar[a], 1);
      ptx::mbar_init(&tempty_bar[a], kEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_h);
    ptx::prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // A kernel launched after this one as a programmatic dependent may be
  // scheduled from now on, on whatever SM resources are free (for another
  // sampling call: the SMs this grid's blocks leave); it must wait for this
  // grid to complete before it reads anything this grid writes.  The top-K
  // modes let their dependent (the list reduction, which can do nothing
  // before this grid ends) be scheduled only as each block finishes.
  if constexpr (!kTopkMode<kMode>) ptx::grid_launch_dependents();
  const uint32_t tmem_base = *tmem_holder;
  const Waiter waiter{abort_flag, p.wait_limit_ns};
  const uint32_t h_bytes = p.h_box_rows * 128u;  // the H box; the W slice follows it

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // The whole warp runs the loop and one elected lane issues the copies.
    // (The same loop run by one lane alone took several times as many cycles
    // per stage whenever the epilogue warps sharing its SM sub-partition were
    // busy, and the stage time followed.)
    {
      const bool issuer = ptx::elect_one();
      const uint64_t pol_w = p.n_mt > 1 ? ptx::policy_evict_normal() : ptx::policy_evict_first();
      const uint64_t pol_h = ptx::policy_evict_last();
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      bool deferring = p.pdl != 0;
      DeferredH defer;
      auto flush_h = [&]() {
        ptx::grid_dependency_wait();
        for (int i = 0; i < defer.n; ++i)
          if (issuer)
            ptx::tma_load_2d(smem + size_t(defer.stage[i]) * p.stage_bytes, &tmap_h,
                             &full_bar[defer.stage[i]], defer.kb[i] * kBlockK, defer.row[i], pol_h);
        defer.n = 0;
        deferring = false;
      };
      for (int unit = blockIdx.x; ok && unit < n_units; unit += gridDim.x) {
        const int vt = unit / p.n_mt, mt = unit % p.n_mt;
        // Each vocabulary block starts its K loop at its own slice, so CTAs
        // working at the same moment read different H lines.  The start
        // depends on the (global) vocabulary block only, so a row's sums (and
        // its sample) do not depend on the batch size or on the sharding.
        const int k_start =
            int((uint32_t(vt + (p.vocab_offset >> 8)) * 5u) % uint32_t(p.n_kb));
        for (int kk = 0; kk < p.n_kb; ++kk) {
          const int kb = kk + k_start < p.n_kb ? kk + k_start : kk + k_start - p.n_kb;
          if (!waiter.wait_warp(&empty_bar[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(stage) * p.stage_bytes;
          if (issuer) {
            ptx::mbar_arrive_expect_tx(&full_bar[stage], h_bytes + kSmemB);
            ptx::tma_load_2d(sa + h_bytes, &tmap_w, &full_bar[stage], kb * kBlockK, vt * kBlockN,
                             pol_w);
          }
          if (deferring) {
            defer.stage[defer.n] = stage;
            defer.kb[defer.n] = kb;
            defer.row[defer.n++] = mt * kBlockM;
          } else if (issuer) {
            ptx::tma_load_2d(sa, &tmap_h, &full_bar[stage], kb * kBlockK, mt * kBlockM, pol_h);
          }
          ++issued;
          if (++stage == p.n_stages) {
            stage = 0;
            phase ^= 1u;
          }
          if (deferring && defer.n == int(p.n_stages)) flush_h();
        }
      }
      if (deferring) flush_h();
      // Every issued copy must land before the CTA (and its shared memory)
      // goes away: wait for the last fill of each stage.
      for (uint32_t s = 0; s < p.n_stages; ++s) {
        const uint32_t fills = issued / p.n_stages + (s < issued % p.n_stages ? 1u : 0u);
        if (fills) waiter.drain(&full_bar[s], (fills - 1u) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // Warp-wide like the producer; one elected lane issues the MMAs and
    // commits.  Stage s's operand descriptors are stage 0's plus s times the
    // stage size / 16 in the start-address field (shared-memory addresses stay
    // below 256 KB, so the 14-bit field never carries), and a K step of 16
    // bf16 (32 bytes) adds 2.
    {
      const bool issuer = ptx::elect_one();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t s0 = ptx::smem_u32(smem);
      const uint64_t desc_a0 = ptx::smem_desc_sw128(s0);
      const uint64_t desc_b0 = ptx::smem_desc_sw128(s0 + h_bytes);
      const uint32_t stage_units = p.stage_bytes >> 4;
      for (int unit = blockIdx.x; ok && unit < n_units; unit += gridDim.x) {
        if (!waiter.wait_warp(&tempty_bar[acc], acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBlockN;
        for (int kb = 0; kb < p.n_kb; ++kb) {
          if (!waiter.wait_warp(&full_bar[stage], phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t off = uint64_t(stage * stage_units);
          if (issuer) {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              ptx::mma_bf16(d_tmem, desc_a0 + off + uint64_t(2 * k),
                            desc_b0 + off + uint64_t(2 * k), kIdesc, (kb | k) != 0 ? 1u : 0u);
            ptx::mma_commit(&empty_bar[stage]);
          }
          __syncwarp();
          if (++stage == p.n_stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (issuer) ptx::mma_commit(&tfull_bar[acc]);
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs must be complete before tensor memory is released.
      if (issuer) ptx::mma_commit(drain_bar);
      __syncwarp();
      waiter.drain(drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    if (p.pdl) ptx::grid_dependency_wait();  // the per-row inputs may still be in flight
    const int e = warp - 2;
    const int quad = warp & 3;  // the tensor-memory lane quadrant this warp may read
    const int half = e >> 2;    // which 128-column half of the unit
    uint32_t acc = 0, acc_phase = 0;
    EpilogueState<kMode> est;
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const int vt = unit / p.n_mt, mt = unit % p.n_mt;
      const int row0 = mt * kBlockM + quad * 32;
      const int tile = vt * 2 + half;
      const bool work = row0 < p.B && tile < p.n_tiles;
      const bool last = unit + int(gridDim.x) >= n_units;
      // This warp's lanes and columns of both accumulator buffers.
      const uint32_t lanes = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(half * kTileV);
      // A CTA's last unit: its noise is made while its W slices stream in.
      const bool ahead = last && work;
      const uint32_t other = lanes + (acc ^ 1u) * kBlockN;
      if (ahead) noise_ahead(p, other, row0 + lane, tile);
      int ok = 0;
      if (lane == 0) ok = waiter.wait(&tfull_bar[acc], acc_phase) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      if (work)
        epilogue_unit<kMode>(p, lanes + acc * kBlockN, row0 + lane, tile, est, other, ahead);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty_bar[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    epilogue_finish<kMode>(p, est);
  }

  ptx::tc_fence_before();
  __threadfence();  // this thread's row-key updates are visible device-wide
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  finish_rows(p);
  if constexpr (kTopkMode<kMode>) ptx::grid_launch_dependents();
}

// ---------------------------------------------------------------------------
// Stage 1 for an even number of 128-row batch blocks: CTA pairs (2-CTA
// clusters) run M = 256, N = 256, K = 16 MMAs (cta_group::2).  A unit is (vocabulary block vt
// of 256 ids, pair block mp of 256 batch rows).  CTA r of the pair loads batch
// rows mp*256 + r*128 .. +127 (its half of A) and vocabulary rows vt*256 +
// r*128 .. +127 (its half of B) into its own shared memory, 32 KB a stage, so
// six stages fit; every copy signals the even ("leader") CTA's full barrier.
// The leader's MMA warp (one elected lane) accumulates into both CTAs' tensor memory
// (rows r*128.. in CTA r, all 256 columns) and multicasts its commits to both
// CTAs' barriers.  Each CTA's epilogue reads its own 128 rows; the leader's
// "tensor memory empty" barrier collects the epilogue warps of both CTAs.
constexpr int kPairStages = 6;
static_assert(kPairStages <= 8, "a ring fill of deferred H copies fits DeferredH");
constexpr uint32_t kPairSmemA = 128 * kBlockK * 2;  // 16 KB: this CTA's batch rows
constexpr uint32_t kPairSmemB = 128 * kBlockK * 2;  // 16 KB: this CTA's vocabulary rows
constexpr uint32_t kPairStageBytes = kPairSmemA + kPairSmemB;
constexpr size_t kPairBarOffset = size_t(kPairStages) * kPairStageBytes;
constexpr size_t kPairSmemBytes = 1024 + kPairBarOffset + 256;
constexpr uint32_t kPairIdesc = ptx::idesc_bf16_f32(2 * kBlockM, kBlockN);
static_assert(kPairSmemBytes <= 232448, "pair kernel shared memory");

// The unit (vocabulary block vt, pair batch block mp) that CTA pair `pair`
// takes k-th; false when it has no more.  Plain order: unit pair + k * n_pairs
// of the vocabulary-major list, so the n_mp units of one vocabulary block run
// on neighbouring pairs at about the same time and all but the first read its
// W tile from L2; a pair's batch block changes from one unit to the next
// unless n_pairs is a multiple of n_mp.  Grouped order (kGrouped, launched by
// the host for the top-K modes when it needs no more waves than the plain
// one): groups of n_mp pairs walk the same vocabulary blocks, pair j of a
// group always on batch block j, so each of its epilogue threads keeps one row
// for the whole call -- one candidate list a thread instead of one a unit;
// the pairs left over take the remaining blocks whole, one batch block after
// the other.  (A separate kernel: the grouped loop in the plain kernels cost
// the sampling modes about 0.5 % and spilled the top-K modes' registers.)
template <bool kGrouped>
__device__ __forceinline__ bool pair_unit(const Stage1Params& p, int pair, int k, int n_pairs,
                                          int n_mp, int n_vt, int& vt, int& mp) {
  if constexpr (kGrouped) {
    const int G = p.pair_groups;
    if (pair < G * n_mp) {
      vt = pair / n_mp + k * G;
      mp = pair % n_mp;
      return k < p.pair_group_blocks && vt < n_vt;
    }
    const int n_left = n_pairs - G * n_mp, l = pair - G * n_mp;
    vt = min(n_vt, G * p.pair_group_blocks) + l + (k / n_mp) * n_left;
    mp = k % n_mp;
    return vt < n_vt;
  } else {
    const int u = pair + k * n_pairs;
    vt = u / n_mp;
    mp = u % n_mp;
    return u < n_vt * n_mp;
  }
}

template <int kMode, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_pair_kernel(const __grid_constant__ CUtensorMap tmap_h,
                       const __grid_constant__ CUtensorMap tmap_w, const Stage1Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kPairBarOffset);
  uint64_t* empty_bar = full_bar + kPairStages;
  uint64_t* tfull_bar = empty_bar + kPairStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = int(ptx::cluster_ctarank());
  const bool leader = rank == 0;
  const int pair_id = int(blockIdx.x) >> 1;
  const int n_pairs = int(gridDim.x) >> 1;
  const int n_mp = (p.B + 2 * kBlockM - 1) / (2 * kBlockM);
  const int n_vt = (p.n_tiles + 1) / 2;  // not from V + 255 (32-bit overflow)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull_bar[a], 1);
      ptx::mbar_init(&tempty_bar[a], 2 * kEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_h);
    ptx::prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {  // one warp in each CTA of the pair, together
    ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before either uses the other's
  ptx::tc_fence_after();
  if constexpr (!kTopkMode<kMode>) ptx::grid_launch_dependents();  // as in stage1_kernel
  const uint32_t tmem_base = *tmem_holder;
  const Waiter waiter{abort_flag, p.wait_limit_ns};

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    // Warp-wide, one elected lane issuing (as in stage1_kernel).
    {
      const bool issuer = ptx::elect_one();
      const uint64_t pol_w = n_mp > 1 ? ptx::policy_evict_normal() : ptx::policy_evict_first();
      const uint64_t pol_h = ptx::policy_evict_last();
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      bool deferring = p.pdl != 0;
      DeferredH defer;
      auto flush_h = [&]() {
        ptx::grid_dependency_wait();
        for (int i = 0; i < defer.n; ++i)
          if (issuer)
            ptx::tma_load_2d_pair(smem + size_t(defer.stage[i]) * kPairStageBytes, &tmap_h,
                                  ptx::cluster_addr(&full_bar[defer.stage[i]], 0),
                                  defer.kb[i] * kBlockK, defer.row[i], pol_h);
        defer.n = 0;
        deferring = false;
      };
      int vt, mp;
      for (int k = 0;
           ok && pair_unit<kGrouped>(p, pair_id, k, n_pairs, n_mp, n_vt, vt, mp); ++k) {
        const int k_start =
            int((uint32_t(vt + (p.vocab_offset >> 8)) * 5u) % uint32_t(p.n_kb));
        // Rows past the end are read from the last valid row instead (their
        // accumulator rows / columns are never used), so no box lies wholly
        // outside its tensor.
        const int a_y = min(mp * 2 * kBlockM + rank * kBlockM, p.B - 1);
        const int w_y = min(vt * kBlockN + rank * (kBlockN / 2), p.V - 1);
        for (int kk = 0; kk < p.n_kb; ++kk) {
          const int kb = kk + k_start < p.n_kb ? kk + k_start : kk + k_start - p.n_kb;
          if (!waiter.wait_warp(&empty_bar[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + size_t(stage) * kPairStageBytes;
          const uint32_t full_addr = ptx::cluster_addr(&full_bar[stage], 0);
          if (issuer) {
            if (leader) ptx::mbar_arrive_expect_tx(&full_bar[stage], 2 * kPairStageBytes);
            ptx::tma_load_2d_pair(sa + kPairSmemA, &tmap_w, full_addr, kb * kBlockK, w_y, pol_w);
          }
          if (deferring) {
            defer.stage[defer.n] = stage;
            defer.kb[defer.n] = kb;
            defer.row[defer.n++] = a_y;
          } else if (issuer) {
            ptx::tma_load_2d_pair(sa, &tmap_h, full_addr, kb * kBlockK, a_y, pol_h);
          }
          ++issued;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (deferring && defer.n == kPairStages) flush_h();
        }
      }
      if (deferring) flush_h();
      // The leader's full barriers see both CTAs' copies land; wait for the
      // last fill of each stage before anything goes away.
      if (leader) {
        for (uint32_t s = 0; s < uint32_t(kPairStages); ++s) {
          const uint32_t fills = issued / kPairStages + (s < issued % kPairStages ? 1u : 0u);
          if (fills) waiter.drain(&full_bar[s], (fills - 1u) & 1u);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA only) ----------------
    // Warp-wide, one elected lane issuing (as in stage1_kernel).
    if (leader) {
      const bool issuer = ptx::elect_one();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t s0 = ptx::smem_u32(smem);
      const uint64_t desc_a0 = ptx::smem_desc_sw128(s0);
      const uint64_t desc_b0 = ptx::smem_desc_sw128(s0 + kPairSmemA);
      int vt, mp;
      for (int k = 0;
           ok && pair_unit<kGrouped>(p, pair_id, k, n_pairs, n_mp, n_vt, vt, mp); ++k) {
        if (!waiter.wait_warp(&tempty_bar[acc], acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBlockN;
        for (int kb = 0; kb < p.n_kb; ++kb) {
          if (!waiter.wait_warp(&full_bar[stage], phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t off = uint64_t(stage * (kPairStageBytes >> 4));
          if (issuer) {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              ptx::mma_bf16_pair(d_tmem, desc_a0 + off + uint64_t(2 * k),
                                 desc_b0 + off + uint64_t(2 * k), kPairIdesc,
                                 (kb | k) != 0 ? 1u : 0u);
            ptx::mma_commit_pair_multicast(&empty_bar[stage], 0x3);
          }
          __syncwarp();
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (issuer) ptx::mma_commit_pair_multicast(&tfull_bar[acc], 0x3);
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (issuer) ptx::mma_commit_pair(drain_bar);
      __syncwarp();
      waiter.drain(drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    if (p.pdl) ptx::grid_dependency_wait();  // the per-row inputs may still be in flight
    const int e = warp - 2;
    const int quad = warp & 3;
    const int half = e >> 2;
    const uint32_t tempty_addr0 = ptx::cluster_addr(&tempty_bar[0], 0);
    const uint32_t tempty_addr1 = ptx::cluster_addr(&tempty_bar[1], 0);
    uint32_t acc = 0, acc_phase = 0;
    EpilogueState<kMode> est;
    int vt, mp;
    for (int k = 0; pair_unit<kGrouped>(p, pair_id, k, n_pairs, n_mp, n_vt, vt, mp); ++k) {
      int ok = 0;
      if (lane == 0) ok = waiter.wait(&tfull_bar[acc], acc_phase) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row0 = mp * 2 * kBlockM + rank * kBlockM + quad * 32;
      const int tile = vt * 2 + half;
      if (row0 < p.B && tile < p.n_tiles) {
        const uint32_t taddr =
            tmem_base + (uint32_t(quad * 32) << 16) + acc * kBlockN + uint32_t(half * kTileV);
        epilogue_unit<kMode>(p, taddr, row0 + lane, tile, est, 0u, false);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc == 0 ? tempty_addr0 : tempty_addr1);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    epilogue_finish<kMode>(p, est);
  }

  ptx::tc_fence_before();
  __threadfence();
  __syncthreads();
  // Both CTAs are done with each other's barriers and the leader's MMAs have
  // drained before the pair's tensor memory is released.
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  ptx::cluster_sync();
  finish_rows(p);
  if constexpr (kTopkMode<kMode>) ptx::grid_launch_dependents();
}

// Diagnostic: the bounded wait of the sampling kernels, on an mbarrier that no
// thread ever arrives on.  It gives up after limit_ns, records the timeout in
// the device error word, and returns -- the path a stalled pipeline takes.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_word;
  ptx::mbar_init(&bar, 1);
  abort_word = 0u;
  ptx::fence_barrier_init();
  const Waiter waiter{&abort_word, limit_ns};
  waiter.wait(&bar, 0);  // phase 0 never completes
}

// Copy n bytes from mapped (pinned) host memory to device memory with SM
// loads over the host link: 16 bytes a thread when both ends are 16-byte
// aligned, else byte by byte.
__global__ void stage_in_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                size_t n, int vec) {
  ptx::grid_launch_dependents();  // the sampling kernel may start streaming W now
  const size_t tid = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  if (vec) {
    const size_t n16 = n / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (size_t i = tid; i < n16; i += stride) d4[i] = s4[i];
    for (size_t i = n16 * 16 + tid; i < n; i += stride) dst[i] = src[i];
  } else {
    for (size_t i = tid; i < n; i += stride) dst[i] = src[i];
  }
}

// The word -> Gumbel transform alone, on given words (diagnostic entry point).
__global__ void gumbel_transform_kernel(const uint32_t* __restrict__ words, int64_t n,
                                        float* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = gumbel_from_word(words[i]);
}

// The noise stage 1 adds, element by element (diagnostic entry point).
__global__ void noise_kernel(const uint64_t* __restrict__ seeds, uint64_t seed, uint64_t offset,
                             int64_t b0, int64_t nb, int64_t v0, int64_t nv,
                             float* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nb * nv) return;
  const int64_t b = b0 + i / nv, v = v0 + i % nv;
  const uint64_t sd = seeds ? seeds[b] : seed;
  const uint4 r = philox4x32_10(
      make_uint4(static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(b),
                 static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32)),
      PhiloxSchedule(sd));
  out[i] = gumbel_from_word(select_word(r, static_cast<uint32_t>(v & 3)));
}

}  // namespace fs
