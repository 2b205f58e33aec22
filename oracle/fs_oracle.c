/*
 * fs_oracle.c -- plain fp64 CPU oracle for fused LM-head + exact Gumbel-max
 * sampling ("FlashSampling: Fast and Memory-Efficient Exact Sampling").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library; the two are independent restatements of the same definition.
 *
 * What it computes, for one row b of the batch (all arithmetic in double):
 *   l[v]   = sum_k H[b,k] * W[v,k]                 (LM-head logits; the
 *            aitrends.kr write-up, "Stage 1 (Fused Kernel)": logits from the
 *            hidden state H and the weight W)
 *   l'[v]  = l[v] / T_b                             (temperature scaling, same
 *            passage); T_b <= 0 or non-finite => greedy: l' = l and no noise
 *   g[v]   = -log(-log u[v])                        (Gumbel noise, same passage)
 *   s[v]   = l'[v] + g[v], or -inf where the vocab mask bit is clear
 *   per vocabulary tile t: m_t = max s, i_t = lowest v attaining m_t
 *            (tomesphere abstract: "keep only one maximizer per row and per
 *            vocabulary tile"), L_t = log sum_{unmasked v in t} exp(l'[v])
 *            (the group log-mass L_k of the tensor-parallel / Group-Gumbel-Max
 *            passages of the aitrends.kr write-up)
 *   sample = lowest v attaining max_v s            (Stage 2, "Reduction")
 *
 * Readings where the pages are silent (the choices this oracle makes):
 *   - the uniform u comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 *     "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) with
 *     key = (seed_b & 0xffffffff, seed_b >> 32),
 *     counter = (v >> 2, b, offset & 0xffffffff, offset >> 32),
 *     and output word (v & 3);
 *   - u = ((w & 0x7fffff) + 0.5) * 2^-23 (the word's low 23 bits), so
 *     0 < u < 1 and u is exact in fp32;
 *   - ties go to the lowest vocabulary index;
 *   - a fully masked tile or row gives m = -inf, index -1, L = -inf;
 *   - for a greedy row L_t is max l over the tile's unmasked entries.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- Philox4x32-10, from the SC'11 definition ---------------------------
 * Round function: with the two multipliers M0, M1, the 4-word counter
 * (x0,x1,x2,x3) and the 2-word key (k0,k1):
 *   (hi0,lo0) = M0 * x0,  (hi1,lo1) = M1 * x2      (64-bit products)
 *   x <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0)
 * Ten rounds; the key is bumped by the Weyl constants (W0, W1) between
 * consecutive rounds. */
static const uint32_t PHILOX_MULT_0 = 0xD2511F53u;
static const uint32_t PHILOX_MULT_1 = 0xCD9E8D57u;
static const uint32_t PHILOX_WEYL_0 = 0x9E3779B9u;
static const uint32_t PHILOX_WEYL_1 = 0xBB67AE85u;

void fso_philox4x32_10(const uint32_t counter[4], const uint32_t key[2],
                       uint32_t out[4]) {
  uint32_t x0 = counter[0], x1 = counter[1], x2 = counter[2], x3 = counter[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_WEYL_0;
      k1 += PHILOX_WEYL_1;
    }
    uint64_t prod0 = (uint64_t)PHILOX_MULT_0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)PHILOX_MULT_1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ x1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ x3 ^ k1;
    uint32_t n3 = lo0;
    x0 = n0; x1 = n1; x2 = n2; x3 = n3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* 32-bit random word -> uniform in (0,1): keep the low 23 bits, centre. */
double fso_uniform(uint32_t word) {
  return ((double)(word & 0x7fffffu) + 0.5) * (1.0 / 8388608.0); /* 2^-23 */
}

/* Gumbel(0,1) by inversion: g = -log(-log u). */
double fso_gumbel(double u) { return -log(-log(u)); }

/* The random word that drives element (b, v) of a call with (seed, offset). */
uint32_t fso_noise_word(uint64_t seed, uint64_t offset, int64_t b, int64_t v) {
  uint32_t counter[4], key[2], out[4];
  counter[0] = (uint32_t)((uint64_t)v >> 2);
  counter[1] = (uint32_t)b;
  counter[2] = (uint32_t)(offset & 0xffffffffu);
  counter[3] = (uint32_t)(offset >> 32);
  key[0] = (uint32_t)(seed & 0xffffffffu);
  key[1] = (uint32_t)(seed >> 32);
  fso_philox4x32_10(counter, key, out);
  return out[(uint64_t)v & 3u];
}

double fso_noise(uint64_t seed, uint64_t offset, int64_t b, int64_t v) {
  return fso_gumbel(fso_uniform(fso_noise_word(seed, offset, b, v)));
}

/* The uniform that merges draw for row b and partition (or online step) k:
 * Philox4x32-10 with the row's key and counter (k >> 2, b | 2^31, offset low,
 * offset high), word k & 3 -- a counter domain the sampling noise never uses
 * (its second counter word is the row, below 2^31), so the choice among
 * partitions is independent of the partitions' own samples. */
double fso_merge_uniform(uint64_t seed, uint64_t offset, int64_t b, int64_t k) {
  uint32_t counter[4], key[2], out[4];
  counter[0] = (uint32_t)((uint64_t)k >> 2);
  counter[1] = (uint32_t)b | 0x80000000u;
  counter[2] = (uint32_t)(offset & 0xffffffffu);
  counter[3] = (uint32_t)(offset >> 32);
  key[0] = (uint32_t)(seed & 0xffffffffu);
  key[1] = (uint32_t)(seed >> 32);
  fso_philox4x32_10(counter, key, out);
  return fso_uniform(out[(uint64_t)k & 3u]);
}

/* Noise for the window rows [b0, b0+nb) x vocab [v0, v0+nv), row-major.
 * seeds (optional) gives one seed per absolute row index. */
void fso_noise_grid(const uint64_t *seeds, uint64_t seed, uint64_t offset,
                    int64_t b0, int64_t nb, int64_t v0, int64_t nv,
                    double *out) {
  for (int64_t i = 0; i < nb; ++i) {
    int64_t b = b0 + i;
    uint64_t sd = seeds ? seeds[b] : seed;
    for (int64_t j = 0; j < nv; ++j)
      out[i * nv + j] = fso_noise(sd, offset, b, v0 + j);
  }
}

/* ---- LM-head logits ----------------------------------------------------- */
static double bf16_to_double(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* l = H[b,:] . W[v,:], summed in index order. */
static double logit(const uint16_t *H, const uint16_t *W, int64_t d,
                    int64_t ldh, int64_t ldw, int64_t b, int64_t v) {
  const uint16_t *h = H + b * ldh;
  const uint16_t *w = W + v * ldw;
  double acc = 0.0;
  for (int64_t k = 0; k < d; ++k) acc += bf16_to_double(h[k]) * bf16_to_double(w[k]);
  return acc;
}

void fso_logits(const uint16_t *H, const uint16_t *W, int64_t B, int64_t d,
                int64_t V, int64_t ldh, int64_t ldw, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < B; ++b)
    for (int64_t v = 0; v < V; ++v) out[b * V + v] = logit(H, W, d, ldh, ldw, b, v);
}

/* ---- the sampling definition, one requested row at a time -------------- */
static int is_greedy(double T) { return !(T > 0.0) || isinf(T); }

static int allowed(const uint32_t *mask, int64_t mask_ld, int64_t b, int64_t v) {
  if (!mask) return 1;
  return (int)((mask[b * mask_ld + v / 32] >> (v % 32)) & 1u);
}

/*
 * For each requested row rows[r] (0 <= rows[r] < B):
 *   out_idx[r]             sampled index (lowest v attaining max s), -1 if
 *                          every entry is masked
 *   out_gap[r]             s(1) - s(2) over the row (+inf with < 2 entries)
 *   tile_max[r*nt + t]     m_t            (-inf for a fully masked tile)
 *   tile_idx[r*nt + t]     i_t            (-1 for a fully masked tile)
 *   tile_lse[r*nt + t]     L_t            (-inf for a fully masked tile)
 *   tile_gap[r*nt + t]     in-tile s(1) - s(2)
 *   logits_out[r*V + v]    l[v]           (optional)
 *   scores_out[r*V + v]    s[v]           (optional)
 * with nt = ceil(V / tile).  Returns 0, or -1 on a bad argument.
 */
int fso_sample_rows(const uint16_t *H, const uint16_t *W, int64_t B, int64_t d,
                    int64_t V, int64_t ldh, int64_t ldw,
                    const float *temperature, const uint32_t *mask,
                    int64_t mask_ld, const uint64_t *seeds, uint64_t seed,
                    uint64_t offset, int64_t tile, const int64_t *rows,
                    int64_t n_rows, int64_t *out_idx, double *out_gap,
                    double *tile_max, int64_t *tile_idx, double *tile_lse,
                    double *tile_gap, double *logits_out, double *scores_out) {
  if (!H || !W || B <= 0 || d <= 0 || V <= 0 || tile <= 0 || ldh < d || ldw < d)
    return -1;
  const int64_t nt = (V + tile - 1) / tile;
  double *l = (double *)malloc(sizeof(double) * (size_t)V);
  double *lp = (double *)malloc(sizeof(double) * (size_t)V);
  double *s = (double *)malloc(sizeof(double) * (size_t)V);
  unsigned char *ok = (unsigned char *)malloc((size_t)V);
  if (!l || !lp || !s || !ok) {
    free(l); free(lp); free(s); free(ok);
    return -1;
  }
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t b = rows ? rows[r] : r;
    if (b < 0 || b >= B) {
      free(l); free(lp); free(s); free(ok);
      return -1;
    }
    const double T = temperature ? (double)temperature[b] : 1.0;
    const int greedy = is_greedy(T);
    const uint64_t sd = seeds ? seeds[b] : seed;

#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < V; ++v) {
      l[v] = logit(H, W, d, ldh, ldw, b, v);
      ok[v] = (unsigned char)allowed(mask, mask_ld, b, v);
      if (greedy) {
        lp[v] = l[v];
        s[v] = l[v];
      } else {
        lp[v] = l[v] / T;
        s[v] = lp[v] + fso_noise(sd, offset, b, v);
      }
      if (isnan(s[v])) ok[v] = 0; /* a NaN score can never be the maximum */
      if (!ok[v]) s[v] = -INFINITY;
    }

    /* per vocabulary tile */
    for (int64_t t = 0; t < nt; ++t) {
      const int64_t lo = t * tile, hi = (lo + tile < V) ? lo + tile : V;
      double best = -INFINITY, second = -INFINITY;
      int64_t arg = -1;
      double lmax = -INFINITY;
      for (int64_t v = lo; v < hi; ++v) {
        if (!ok[v]) continue;
        if (arg < 0 || s[v] > best) {
          second = best;
          best = s[v];
          arg = v;
        } else if (s[v] > second) {
          second = s[v];
        }
        if (lp[v] > lmax) lmax = lp[v];
      }
      double lse;
      if (arg < 0) {
        lse = -INFINITY;
      } else if (greedy) {
        lse = lmax;
      } else {
        double acc = 0.0;
        for (int64_t v = lo; v < hi; ++v)
          if (ok[v]) acc += exp(lp[v] - lmax);
        lse = lmax + log(acc);
      }
      if (tile_max) tile_max[r * nt + t] = best;
      if (tile_idx) tile_idx[r * nt + t] = arg;
      if (tile_lse) tile_lse[r * nt + t] = lse;
      if (tile_gap) tile_gap[r * nt + t] = (arg < 0) ? INFINITY : best - second;
    }

    /* the whole row */
    {
      double best = -INFINITY, second = -INFINITY;
      int64_t arg = -1;
      for (int64_t v = 0; v < V; ++v) {
        if (!ok[v]) continue;
        if (arg < 0 || s[v] > best) {
          second = best;
          best = s[v];
          arg = v;
        } else if (s[v] > second) {
          second = s[v];
        }
      }
      if (out_idx) out_idx[r] = arg;
      if (out_gap) out_gap[r] = (arg < 0) ? INFINITY : best - second;
    }
    if (logits_out) memcpy(logits_out + r * V, l, sizeof(double) * (size_t)V);
    if (scores_out) memcpy(scores_out + r * V, s, sizeof(double) * (size_t)V);
  }
  free(l); free(lp); free(s); free(ok);
  return 0;
}

/* Threads an OpenMP parallel region of this library uses (1 without OpenMP),
 * and a setter for it (timing only; the results do not depend on it). */
#ifdef _OPENMP
#include <omp.h>
int fso_num_threads(void) { return omp_get_max_threads(); }
void fso_set_num_threads(int n) { if (n > 0) omp_set_num_threads(n); }
#else
int fso_num_threads(void) { return 1; }
void fso_set_num_threads(int n) { (void)n; }
#endif
