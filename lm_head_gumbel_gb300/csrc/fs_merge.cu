// fs_merge.cu -- combining per-partition sampling results.
//
// FlashSampling's exactness arguments (tomesphere abstract: the kernel is exact
// because argmax decomposes over partitions; grouped variants for online and
// tensor-parallel settings are exact by hierarchical factorisation of the
// categorical; aitrends.kr write-up, tensor-parallel and Group-Gumbel-Max
// paragraphs) turn into three small kernels:
//   row_lse_kernel      the row's log-mass L = log sum_t exp(L_t) from the
//                       stage-1 kernel's per-tile log-masses;
//   group_merge_kernel  one sample per row from P partitions' (z_k, m_k, L_k):
//                       exact (argmax_k m_k) or Group-Gumbel-Max
//                       (argmax_k L_k + G_k, fresh Gumbel noise);
//   online_merge_kernel the O(1)-state binary merge rule with a Bernoulli
//                       switch, one group at a time;
//   topk_reduce_kernel  each row's K best of its per-tile top-K candidates.
// The merges' own randomness uses Philox on a counter domain the sampling noise
// never uses (second counter word = row | 2^31), keyed by the row's seed.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fs_noise.cuh"
#include "fs_sample.h"

namespace fs {
namespace {

constexpr int kLseThreads = 128;
constexpr int kMergeThreads = 128;

__device__ __forceinline__ float block_reduce(float v, bool is_max) {
  __shared__ float part[kLseThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();  // part[] may still be read by a previous call
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = part[0];
#pragma unroll
  for (int w = 1; w < kLseThreads / 32; ++w) r = is_max ? fmaxf(r, part[w]) : r + part[w];
  return r;
}

// One block per row.  Greedy rows (T <= 0, NaN or inf) report the largest
// tile value, i.e. the row's largest logit, matching the per-tile convention.
__global__ void __launch_bounds__(kLseThreads)
    row_lse_kernel(const float* __restrict__ tile_lse, const float* __restrict__ temperature,
                   int32_t n_tiles, float* __restrict__ out_lse) {
  const int row = blockIdx.x;
  const float* t = tile_lse + int64_t(row) * n_tiles;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < n_tiles; i += kLseThreads) m = fmaxf(m, t[i]);
  m = block_reduce(m, true);
  const float T = temperature ? temperature[row] : 1.0f;
  const bool greedy = !(T > 0.0f) || isinf(T);
  if (greedy || m == -INFINITY) {
    if (threadIdx.x == 0) out_lse[row] = m;
    return;
  }
  float s = 0.0f;
  for (int i = threadIdx.x; i < n_tiles; i += kLseThreads) s += expf(t[i] - m);
  s = block_reduce(s, false);
  if (threadIdx.x == 0) out_lse[row] = m + logf(s);
}

__device__ __forceinline__ uint32_t merge_word(const PhiloxSchedule& ks, uint64_t offset, int b,
                                               uint32_t k) {
  const uint4 r = philox4x32_10(make_uint4(k >> 2, static_cast<uint32_t>(b) | 0x80000000u,
                                           static_cast<uint32_t>(offset),
                                           static_cast<uint32_t>(offset >> 32)),
                                ks);
  return select_word(r, k & 3u);
}

// One thread per row.
__global__ void __launch_bounds__(kMergeThreads)
    group_merge_kernel(const int64_t* __restrict__ z, const float* __restrict__ m,
                       const float* __restrict__ L, int32_t P, int32_t B, int mode,
                       const uint64_t* __restrict__ seeds, uint64_t seed, uint64_t offset,
                       int64_t* __restrict__ out_idx, float* __restrict__ out_L) {
  const int b = blockIdx.x * kMergeThreads + threadIdx.x;
  if (b >= B) return;
  const PhiloxSchedule ks(seeds ? seeds[b] : seed);
  float best = -INFINITY;
  int64_t pick = -1;
  float lmax = -INFINITY;
  for (int k = 0; k < P; ++k) {
    const int64_t i = int64_t(k) * B + b;
    const int64_t zk = z[i];
    float key;
    bool valid = zk >= 0;
    if (mode == FS_MERGE_EXACT) {
      key = m[i];
    } else {
      const float Lk = L[i];
      valid = valid && Lk > -INFINITY;
      key = Lk + gumbel_from_word(merge_word(ks, offset, b, uint32_t(k)));
    }
    if (valid && key > best) {
      best = key;
      pick = zk;
    }
    if (L != nullptr) lmax = fmaxf(lmax, L[i]);
  }
  out_idx[b] = pick;
  if (out_L != nullptr) {
    float r = lmax;
    if (lmax > -INFINITY) {
      float s = 0.0f;
      for (int k = 0; k < P; ++k) s += expf(L[int64_t(k) * B + b] - lmax);
      r = lmax + logf(s);
    }
    out_L[b] = r;
  }
}

__global__ void __launch_bounds__(kMergeThreads)
    online_merge_kernel(int64_t* __restrict__ state_z, float* __restrict__ state_L,
                        const int64_t* __restrict__ new_z, const float* __restrict__ new_L,
                        int32_t B, uint64_t step, const uint64_t* __restrict__ seeds,
                        uint64_t seed, uint64_t offset) {
  const int b = blockIdx.x * kMergeThreads + threadIdx.x;
  if (b >= B) return;
  const int64_t nz = new_z[b];
  const float nL = new_L[b];
  if (nz < 0 || !(nL > -INFINITY)) return;
  const float sL = state_L[b];
  if (state_z[b] < 0 || !(sL > -INFINITY)) {  // empty state: take the group
    state_z[b] = nz;
    state_L[b] = nL;
    return;
  }
  const float hi = fmaxf(sL, nL), lo = fminf(sL, nL);
  const float Lp = hi + log1pf(expf(lo - hi));  // logaddexp
  const PhiloxSchedule ks(seeds ? seeds[b] : seed);
  const float u = uniform_from_word(merge_word(ks, offset, b, uint32_t(step)));
  if (u < expf(nL - Lp)) state_z[b] = nz;
  state_L[b] = Lp;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The order of (score, id) candidates: higher score first, then lower id; an
// id of -1 (no candidate) comes after everything.
__device__ __forceinline__ bool precedes(float as, int32_t ai, float bs, int32_t bi) {
  return ai >= 0 && (bi < 0 || as > bs || (as == bs && ai < bi));
}

constexpr int kTopkThreads = 256;

// An order-preserving map of non-NaN floats to unsigned integers, and back.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Merge a sorted list c into the sorted list l, keeping the KC best: the
// better of l[q] and c[KC-1-q] for every q is a bitonic sequence holding the
// KC best of both, which a bitonic merge network sorts.
template <int KC>
__device__ __forceinline__ void list_merge(float (&ls)[KC], int32_t (&li)[KC],
                                           const float (&cs)[KC], const int32_t (&ci)[KC]) {
#pragma unroll
  for (int q = 0; q < KC; ++q) {
    const bool take = precedes(cs[KC - 1 - q], ci[KC - 1 - q], ls[q], li[q]);
    ls[q] = take ? cs[KC - 1 - q] : ls[q];
    li[q] = take ? ci[KC - 1 - q] : li[q];
  }
#pragma unroll
  for (int st = KC / 2; st > 0; st >>= 1) {
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      if ((q & st) != 0) continue;
      const int r = q + st;
      const bool sw = precedes(ls[r], li[r], ls[q], li[q]);
      const float a = ls[q], b = ls[r];
      const int32_t ia = li[q], ib = li[r];
      ls[q] = sw ? b : a;
      ls[r] = sw ? a : b;
      li[q] = sw ? ib : ia;
      li[r] = sw ? ia : ib;
    }
  }
}

// K rounds over the lanes' sorted lists: the best head of the warp, which its
// holder pops.  Every lane receives the round's winner.
template <int KC, typename Emit>
__device__ __forceinline__ void warp_select(float (&ls)[KC], int32_t (&li)[KC], int K,
                                            Emit emit) {
  for (int j = 0; j < K; ++j) {
    float bs = ls[0];
    int32_t bi = li[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float os = __shfl_xor_sync(0xFFFFFFFFu, bs, off);
      const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (precedes(os, oi, bs, bi)) {
        bs = os;
        bi = oi;
      }
    }
    emit(j, bs, bi);
    if (li[0] >= 0 && li[0] == bi) {  // ids are distinct: this lane held the winner
#pragma unroll
      for (int q = 0; q < KC - 1; ++q) {
        ls[q] = ls[q + 1];
        li[q] = li[q + 1];
      }
      ls[KC - 1] = -INFINITY;
      li[KC - 1] = -1;
    }
  }
}

// Every list of one row merged into the row's K best (the fallback of
// topk_reduce_kernel below).  Every slot holds a list sorted best first (an
// empty list starts with id -1).  A thread reads the heads of 8 of its slots
// at once, loads a whole list (16-byte loads) only when its head makes the
// thread's own KC-best list, and merges it by a bitonic network.  Then each
// warp picks its K best by shuffles, and warp 0 picks the row's K best from
// the warps' lists.
template <int KC>
__device__ __noinline__ void merge_all_lists(const float* __restrict__ cand_score,
                                             const int32_t* __restrict__ cand_idx,
                                             int32_t n_tiles, int32_t K,
                                             int64_t* __restrict__ out_idx,
                                             float* __restrict__ out_score, int row) {
  static_assert(KC % 4 == 0, "lists are read 4 entries at a time");
  constexpr int kWarps = kTopkThreads / 32;
  constexpr int kGroup = 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t base = int64_t(row) * n_tiles * KC;
  float ls[KC];
  int32_t li[KC];
#pragma unroll
  for (int q = 0; q < KC; ++q) {
    ls[q] = -INFINITY;
    li[q] = -1;
  }
  for (int t0 = threadIdx.x; t0 < n_tiles; t0 += kTopkThreads * kGroup) {
    float hs[kGroup];
    int32_t hi[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const int t = t0 + g * kTopkThreads;
      hs[g] = -INFINITY;
      hi[g] = -1;
      if (t < n_tiles) {
        hs[g] = cand_score[base + int64_t(t) * KC];
        hi[g] = cand_idx[base + int64_t(t) * KC];
      }
    }
#pragma unroll 1
    for (int g = 0; g < kGroup; ++g) {
      float h_s = hs[0];  // hs[g] by selects: a dynamic index would go to local memory
      int32_t h_i = hi[0];
#pragma unroll
      for (int x = 1; x < kGroup; ++x) {
        h_s = g == x ? hs[x] : h_s;
        h_i = g == x ? hi[x] : h_i;
      }
      if (!precedes(h_s, h_i, ls[KC - 1], li[KC - 1])) continue;
      const int64_t o = base + int64_t(t0 + g * kTopkThreads) * KC;
      const float4* s4 = reinterpret_cast<const float4*>(cand_score + o);
      const int4* i4 = reinterpret_cast<const int4*>(cand_idx + o);
      float cs[KC];
      int32_t ci[KC];
#pragma unroll
      for (int q = 0; q < KC / 4; ++q) {
        const float4 a = s4[q];
        const int4 b = i4[q];
        cs[4 * q] = a.x, cs[4 * q + 1] = a.y, cs[4 * q + 2] = a.z, cs[4 * q + 3] = a.w;
        ci[4 * q] = b.x, ci[4 * q + 1] = b.y, ci[4 * q + 2] = b.z, ci[4 * q + 3] = b.w;
      }
      list_merge<KC>(ls, li, cs, ci);
    }
  }
  // Each warp's K best, by shuffles.
  __shared__ float ws[kWarps][KC];
  __shared__ int32_t wi[kWarps][KC];
  warp_select<KC>(ls, li, K, [&](int j, float bs, int32_t bi) {
    if (lane == 0) {
      ws[warp][j] = bs;
      wi[warp][j] = bi;
    }
  });
  __syncthreads();
  if (warp != 0) return;
  // The row's K best from the warps' lists (lane w holds warp w's).
#pragma unroll
  for (int q = 0; q < KC; ++q) {
    const bool has = lane < kWarps && q < K;
    ls[q] = has ? ws[lane][q] : -INFINITY;
    li[q] = has ? wi[lane][q] : -1;
  }
  warp_select<KC>(ls, li, K, [&](int j, float bs, int32_t bi) {
    if (lane == 0) {
      out_idx[int64_t(row) * K + j] = bi;
      if (out_score != nullptr) out_score[int64_t(row) * K + j] = bi >= 0 ? bs : -INFINITY;
    }
  });
}

constexpr int kSurvivorCap = 256;

// Each row's K best of its candidate lists (Gumbel-top-k: K draws without
// replacement, in draw order).  One block per row.  Two lower bounds of the
// row's K-th best score: the K-th best of the threads' best list heads (K
// distinct entries reach it), and the largest K-th entry of a list (that list
// alone holds K entries reaching it).  Only entries reaching tau, the larger
// bound, can be among the row's K best, and only lists whose head reaches tau
// hold any: the block gathers those entries (at the Qwen3-8B head, K and a
// few more) into shared memory and ranks them (score descending, id
// ascending).  A row where more than kSurvivorCap entries reach tau (many
// equal scores, or fewer than K entries in all) merges all its lists
// instead.  Launched as a programmatic dependent of the stage-1 kernel, which
// lets it start as its blocks finish; it reads the lists only after the
// stage-1 grid has completed.
template <int KC>
__global__ void __launch_bounds__(kTopkThreads)
    topk_reduce_kernel(const float* __restrict__ cand_score,
                       const int32_t* __restrict__ cand_idx, int32_t n_tiles, int32_t K,
                       int64_t* __restrict__ out_idx, float* __restrict__ out_score) {
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ float s_part[kWarps];
  __shared__ int s_n;
  __shared__ float s_score[kSurvivorCap];
  __shared__ int32_t s_id[kSurvivorCap];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the stage-1 grid is complete
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t base = int64_t(row) * n_tiles * KC;
  if (threadIdx.x == 0) {
    s_n = 0;
  }
  __syncthreads();
  // Each thread's best list head, and the largest K-th entry of a list: the
  // heads and K-th entries of kGroup slots are loaded at once.
  constexpr int kGroup = 8;
  float tau = -INFINITY;
  float hb = -INFINITY;
  int32_t hbi = -1;
  int32_t hid0[kGroup];
  float hs0[kGroup];
  for (int t0 = threadIdx.x; t0 < n_tiles; t0 += kTopkThreads * kGroup) {
    int32_t hid[kGroup];
    float hs[kGroup], hk[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const int t = t0 + g * kTopkThreads;
      hid[g] = -1;
      hs[g] = hk[g] = -INFINITY;
      if (t < n_tiles) {
        const int64_t o = base + int64_t(t) * KC;
        hid[g] = cand_idx[o];
        hs[g] = cand_score[o];
        hk[g] = cand_score[o + (K - 1)];
      }
    }
    if (t0 == int(threadIdx.x)) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        hid0[g] = hid[g];
        hs0[g] = hs[g];
      }
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      if (hid[g] < 0) continue;
      tau = fmaxf(tau, hk[g]);
      if (precedes(hs[g], hid[g], hb, hbi)) {
        hb = hs[g];
        hbi = hid[g];
      }
    }
  }
  if (int(threadIdx.x) >= n_tiles) {
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      hid0[g] = -1;
      hs0[g] = -INFINITY;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tau = fmaxf(tau, __shfl_xor_sync(0xFFFFFFFFu, tau, off));
  if (lane == 0) s_part[warp] = tau;
  // The largest score that at least K of the threads' best heads reach (K
  // distinct entries reach it), by bisection over the order-preserving
  // integer image of the scores, one block-wide count per step.  It stops
  // when the interval is 2^11 images wide (a relative width of about 2^-12):
  // its lower end still has K heads reaching it and lets few more entries by.
  const uint32_t my = hbi >= 0 ? order_key(hb) : 0u;  // no head: below every score
  uint32_t lo = 0u, hi = 0xFFFFFFFFu;
  while (hi - lo > (1u << 11)) {
    const uint32_t mid = lo + ((hi - lo) >> 1) + 1u;
    if (__syncthreads_count(my >= mid) >= K)
      lo = mid;
    else
      hi = mid - 1u;
  }
  tau = lo <= order_key(-INFINITY) ? -INFINITY : key_score(lo);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tau = fmaxf(tau, s_part[w]);
  // The entries reaching tau, from the lists whose head reaches it (the heads
  // of the first group are still in registers).
  for (int t0 = threadIdx.x; t0 < n_tiles; t0 += kTopkThreads * kGroup) {
    if (t0 != int(threadIdx.x)) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int t = t0 + g * kTopkThreads;
        hid0[g] = -1;
        hs0[g] = -INFINITY;
        if (t < n_tiles) {
          hid0[g] = cand_idx[base + int64_t(t) * KC];
          hs0[g] = cand_score[base + int64_t(t) * KC];
        }
      }
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      if (hid0[g] < 0 || !(hs0[g] >= tau)) continue;
      const int64_t o = base + int64_t(t0 + g * kTopkThreads) * KC;
      const float4* s4 = reinterpret_cast<const float4*>(cand_score + o);
      const int4* i4 = reinterpret_cast<const int4*>(cand_idx + o);
#pragma unroll
      for (int q4 = 0; q4 < KC / 4; ++q4) {
        const float4 a4 = s4[q4];
        const int4 b4 = i4[q4];
        const float cs[4] = {a4.x, a4.y, a4.z, a4.w};
        const int32_t ci[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (ci[q] >= 0 && cs[q] >= tau) {  // lists are sorted, so these come first
            const int pos = atomicAdd(&s_n, 1);
            if (pos < kSurvivorCap) {
              s_score[pos] = cs[q];
              s_id[pos] = ci[q];
            }
          }
        }
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  if (n > kSurvivorCap) {  // block-uniform
    merge_all_lists<KC>(cand_score, cand_idx, n_tiles, K, out_idx, out_score, row);
    return;
  }
  for (int i = threadIdx.x; i < n; i += kTopkThreads) {
    const float si = s_score[i];
    const int32_t ii = s_id[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += precedes(s_score[j], s_id[j], si, ii) ? 1 : 0;
    if (rank < K) {
      out_idx[int64_t(row) * K + rank] = ii;
      if (out_score != nullptr) out_score[int64_t(row) * K + rank] = si;
    }
  }
  for (int r = n + threadIdx.x; r < K; r += kTopkThreads) {  // fewer candidates than K
    out_idx[int64_t(row) * K + r] = -1;
    if (out_score != nullptr) out_score[int64_t(row) * K + r] = -INFINITY;
  }
}

}  // namespace

fs_status launch_topk_reduce(const float* cand_score, const int32_t* cand_idx, int64_t B,
                             int64_t n_tiles, int64_t cap, int64_t K, int64_t* out_idx,
                             float* out_score, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B), 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (cap == 4)
    e = cudaLaunchKernelEx(&cfg, topk_reduce_kernel<4>, cand_score, cand_idx, int32_t(n_tiles),
                           int32_t(K), out_idx, out_score);
  else
    e = cudaLaunchKernelEx(&cfg, topk_reduce_kernel<16>, cand_score, cand_idx, int32_t(n_tiles),
                           int32_t(K), out_idx, out_score);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

fs_status launch_row_lse(const float* tile_lse, const float* temperature, int64_t B,
                         int64_t n_tiles, float* out_lse, cudaStream_t stream) {
  row_lse_kernel<<<unsigned(B), kLseThreads, 0, stream>>>(tile_lse, temperature,
                                                          int32_t(n_tiles), out_lse);
  if (cudaGetLastError() != cudaSuccess) return FS_ERR_CUDA;
  return FS_OK;
}

}  // namespace fs

extern "C" fs_status fs_group_merge(const int64_t* z, const float* m, const float* L, int64_t P,
                                    int64_t B, int mode, const uint64_t* seeds, uint64_t seed,
                                    uint64_t offset, int64_t* out_idx, float* out_L,
                                    void* stream) {
  using fs::aligned;
  if (!z || !out_idx || P < 1 || B < 1 || B > 65535 || P > (int64_t(1) << 24))
    return FS_ERR_INVALID_ARG;
  if (mode == FS_MERGE_EXACT ? !m : mode == FS_MERGE_GROUP_GUMBEL ? !L : true)
    return FS_ERR_INVALID_ARG;
  if (out_L && !L) return FS_ERR_INVALID_ARG;
  if (!aligned(z, 8) || !aligned(out_idx, 8) || (m && !aligned(m, 4)) || (L && !aligned(L, 4)) ||
      (out_L && !aligned(out_L, 4)) || (seeds && !aligned(seeds, 8)))
    return FS_ERR_INVALID_ARG;
  const int blocks = int((B + fs::kMergeThreads - 1) / fs::kMergeThreads);
  fs::group_merge_kernel<<<blocks, fs::kMergeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      z, m, L, int32_t(P), int32_t(B), mode, seeds, seed, offset, out_idx, out_L);
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

extern "C" fs_status fs_online_merge(int64_t* state_z, float* state_L, const int64_t* new_z,
                                     const float* new_L, int64_t B, uint64_t step,
                                     const uint64_t* seeds, uint64_t seed, uint64_t offset,
                                     void* stream) {
  using fs::aligned;
  if (!state_z || !state_L || !new_z || !new_L || B < 1 || B > 65535 ||
      step > uint64_t(0xFFFFFFFFu))
    return FS_ERR_INVALID_ARG;
  if (!aligned(state_z, 8) || !aligned(new_z, 8) || !aligned(state_L, 4) ||
      !aligned(new_L, 4) || (seeds && !aligned(seeds, 8)))
    return FS_ERR_INVALID_ARG;
  const int blocks = int((B + fs::kMergeThreads - 1) / fs::kMergeThreads);
  fs::online_merge_kernel<<<blocks, fs::kMergeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      state_z, state_L, new_z, new_L, int32_t(B), step, seeds, seed, offset);
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}
