/*
 * fs_sample.h -- C ABI of the fused LM-head + exact Gumbel-max sampler
 * (FlashSampling) for NVIDIA GB300 (sm_103a).
 *
 * What one call computes, per batch row b (tomesphere.com, "FlashSampling:
 * Fast and Memory-Efficient Exact Sampling", Abstract; aitrends.kr write-up,
 * "Stage 1 (Fused Kernel)" and "Stage 2 (Reduction)"):
 *
 *   l[b,v]  = sum_k H[b,k] W[v,k]             LM-head logits, fp32 accumulate
 *   l'[b,v] = l[b,v] / T_b                    temperature scaling
 *   s[b,v]  = l'[b,v] + g[b,v]                Gumbel noise g = -log(-log u)
 *             (-inf where the vocabulary mask clears v)
 *   tile t = 128 consecutive vocabulary ids:  m_t = max s, i_t = argmax s,
 *             L_t = log sum exp(l') over the tile's unmasked ids (optional)
 *   out_idx[b] = the id of max_t m_t          the sampled token
 *
 * The [B,V] logits never reach device memory: they live in the tensor-memory
 * accumulator of one fused kernel; each tile's winner is folded into a per-row
 * maximum in the workspace, and the last CTA to finish writes out_idx.
 * By the Gumbel-max identity the result is an exact sample of
 * softmax(l'[b,:]) restricted to the unmasked ids (aitrends.kr write-up,
 * Gumbel-Max paragraph; exactness over tiles because the argmax decomposes
 * over partitions).
 *
 * Conventions fixed by this library where the pages are silent:
 *   - uniforms: Philox4x32-10 (Salmon et al., SC'11), key = (seed_b low word,
 *     seed_b high word), counter = (v >> 2, b, offset low word, offset high
 *     word), output word v & 3; u = ((word & 0x7fffff) + 0.5) * 2^-23 in (0,1);
 *   - T_b <= 0, NaN or +inf selects greedy decoding for row b: s = l, no noise;
 *   - ties go to the lowest vocabulary index, inside a tile and across tiles;
 *   - a fully masked tile reports m = -inf, i = -1, L = -inf; a fully masked
 *     row samples -1;
 *   - for a greedy row, L_t is the tile's largest unmasked logit.
 *
 * Memory: every pointer in fs_sample_args is a DEVICE pointer owned by the
 * caller; the library allocates no device memory per call.  Calls are
 * asynchronous on the given stream and never synchronise it.
 *
 * Workspace: calls that sample (out_idx != NULL) need fs_workspace_size(B, V)
 * bytes of device workspace that is all-zero before the first call that uses
 * it (e.g. cudaMemset once after allocating).  Every call returns it to
 * all-zero, including a call that ends with a device-side timeout, so it can
 * be reused call after call.  Two calls that may run at the same time (on
 * different streams) need different workspaces.
 */
#ifndef FS_SAMPLE_H_
#define FS_SAMPLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Vocabulary ids per output tile (the per-tile outputs are [B, ceil(V/128)]). */
#define FS_TILE 128

typedef enum fs_status {
  FS_OK = 0,
  FS_ERR_INVALID_ARG = 1,    /* rejected on the host; nothing was launched   */
  FS_ERR_UNSUPPORTED = 2,    /* device is not sm_103 (GB300), or no device    */
  FS_ERR_CUDA = 3,           /* a CUDA runtime/driver call or launch failed   */
  FS_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out           */
  FS_ERR_WORKSPACE = 5       /* workspace missing, too small or misaligned    */
} fs_status;

typedef struct fs_sample_args {
  /* bf16 [B, d] hidden states, row stride ldh elements.  16-byte aligned base,
   * ldh % 8 == 0, ldh >= d. */
  const void *H;
  /* bf16 [V, d] LM-head weight (nn.Linear layout: one row per token), row
   * stride ldw elements.  16-byte aligned base, ldw % 8 == 0, ldw >= d. */
  const void *W;
  /* fp32 [B] per-row temperature, or NULL for T = 1 on every row. */
  const float *temperature;
  /* uint32 [B, mask_ld] packed allow-bits (bit v % 32 of word v / 32 set =
   * token v may be sampled), or NULL for no mask.  mask_ld >= ceil(V/32). */
  const uint32_t *vocab_mask;
  int64_t mask_ld;
  /* uint64 [B] per-row Philox seeds, or NULL to use `seed` on every row. */
  const uint64_t *seeds;
  uint64_t seed;
  /* Philox counter high words; a decoder advances it once per step. */
  uint64_t offset;
  int64_t B, d, V, ldh, ldw;
  /* int64 [B]: sampled token id per row (-1: row fully masked).  May be NULL
   * when out_tile_max/out_tile_idx are given: the call then runs stage 1 only
   * and leaves the per-tile summaries for the caller to merge (e.g. across
   * vocabulary partitions, the aitrends.kr write-up's tensor-parallel and
   * Group-Gumbel-Max paragraphs). */
  int64_t *out_idx;
  /* Optional per-tile outputs, each [B, ceil(V/128)] row-major, or NULL.
   * out_tile_max and out_tile_idx are either both given or both NULL;
   * out_tile_lse (given => the kernel also computes L_t) needs them. */
  float *out_tile_max;
  int32_t *out_tile_idx;
  float *out_tile_lse;
  /* Device workspace, 256-byte aligned, at least fs_workspace_size(B, V)
   * bytes, all-zero before its first use (see "Workspace" above); required
   * when out_idx is given, ignored otherwise. */
  void *workspace;
  size_t workspace_bytes;
  /* Global vocabulary id of W's first row (a multiple of 4, >= 0, with
   * vocab_offset + V < 2^31): a call on a shard of the vocabulary reports
   * global ids (out_idx, out_tile_idx) and draws the noise of the global ids,
   * so the exact merge of the shards' samples (fs_group_merge) is the sample of
   * the unsharded call.  0 for an unsharded call. */
  int64_t vocab_offset;
  /* Optional fp32 [B]: the row's largest noisy score m = max_v s[b,v]
   * (-inf for a fully masked row); needs out_idx. */
  float *out_max;
  /* Optional fp32 [B]: the row's log-mass L = log sum exp(l'[b,v]) over the
   * call's unmasked ids (the group log-mass L_k of the aitrends.kr write-up's
   * tensor-parallel and Group-Gumbel-Max paragraphs; the largest logit for a
   * greedy row); needs out_tile_lse.  Adds a small second kernel. */
  float *out_lse;
  /* FS_FLAG_* bits, 0 for none; unknown bits are FS_ERR_INVALID_ARG. */
  uint32_t flags;
} fs_sample_args;

/*
 * flags: overlap the kernel launched before this call on the same stream (a
 * programmatic dependent launch).  The sampling kernel may then start while
 * that kernel is still running, as its thread blocks leave SMs free, and
 * stream the first slices of W into its shared-memory pipeline; it reads H,
 * the temperatures, seeds and mask, and reads or writes the workspace and
 * every output, only after the earlier kernel has completed and its writes
 * are visible.  So the earlier kernel may produce H and the per-row inputs,
 * but must not write W.  It hides the sampler's launch and pipeline fill
 * behind the kernel that computes H (e.g. the final normalisation of a decode
 * step).  When the earlier work on the stream is not a kernel, the call runs
 * as without the flag.  The results are the same with or without it.  Used by
 * fs_sample, fs_sample_noalloc, fs_sample_host (whose own copy kernel already
 * overlaps it when in_bytes > 0) and fs_sample_topk.  The library's sampling
 * kernels allow such a dependent to be scheduled as soon as they start.
 */
#define FS_FLAG_OVERLAP_PREVIOUS 1u

/* Number of 128-wide vocabulary tiles, ceil(V / 128); 0 for V <= 0. */
int64_t fs_num_tiles(int64_t V);

/* Bytes of workspace a sampling call needs: 256 + 8 * B (a CTA ticket and one
 * 64-bit running maximum per row), rounded up to 256.  Returns 0 for
 * non-positive sizes. */
size_t fs_workspace_size(int64_t B, int64_t V);

/*
 * Sample one token per row (the computation above) on `stream` (a
 * cudaStream_t; NULL = the legacy default stream).  Arguments are checked on
 * the host first: on FS_ERR_INVALID_ARG / FS_ERR_WORKSPACE / FS_ERR_UNSUPPORTED
 * nothing is launched and no output is written.  FS_ERR_CUDA reports a failed
 * launch.  Limits: 1 <= B <= 65535, 1 <= d, 1 <= V < 2^31.
 * Deterministic: identical inputs, seeds and offset give identical outputs on
 * every call, stream and graph replay.
 */
fs_status fs_sample(const fs_sample_args *args, void *stream);

/* Size of the library's built-in scratch array used by fs_sample_noalloc:
 * enough for B <= 8160 rows. */
#define FS_NOALLOC_SCRATCH_BYTES ((size_t)64 << 10) /* 64 KiB */

/*
 * fs_sample for callers that cannot allocate device memory.  (The FlashSampling
 * pages have no counterpart to this entry point; it is a deployment aid.)
 *
 * Some callers cannot call cudaMalloc: a sampler plugged into an inference
 * engine that reserves the whole device for its own memory pool and hands its
 * plugins no allocator, or a decode loop that cannot afford cudaMalloc's
 * implicit device synchronisation.  This entry point computes exactly what
 * fs_sample computes, but instead of args->workspace (ignored, like
 * args->workspace_bytes) it uses a scratch array of FS_NOALLOC_SCRATCH_BYTES
 * that lives inside the library: a file-scope __device__ array that every GPU
 * which loads the library holds until the process exits.  The caller still
 * owns and passes every input and output.  The library calls no cudaMalloc,
 * cudaFree or other allocating routine on this path.
 *
 * - Limit: a sampling call (out_idx given) needs fs_workspace_size(B, V) <=
 *   FS_NOALLOC_SCRATCH_BYTES, i.e. B <= 8160; larger batches return
 *   FS_ERR_WORKSPACE before anything is launched.  Calls that only write
 *   per-tile outputs use no scratch.
 * - Set-up: the first call on a device (with that device current) looks up the
 *   array's device address and clears the array once, with a memset (not an
 *   allocation) enqueued on that call's stream ahead of its kernel, so the
 *   first call may come on any stream, blocking or not; make that first call
 *   before any stream capture.
 * - Sharing: every call on a device uses the same array.  The array must be
 *   all-zero when a call starts, and every call leaves it all-zero.  Calls that
 *   overlap on the GPU (concurrent streams) race on it; serialise them.
 */
fs_status fs_sample_noalloc(const fs_sample_args *args, void *stream);

/* Waits of fs_sample_host. */
#define FS_SYNC_NONE 0   /* return once the work is enqueued                          */
#define FS_SYNC_STREAM 1 /* return after the stream has finished                      */
#define FS_SYNC_IDS 2    /* return as soon as all ids are in host_out (the kernel may  */
                         /* still be winding down; later work on the stream follows it) */

/*
 * One decode step from host memory: the end-to-end form of fs_sample, in one
 * call.  Enqueues on `stream`, in order: a copy of in_bytes from host_in (host
 * memory; pinned, for the copy to be asynchronous) to dev_in (device memory),
 * the fs_sample call described by args -- whose input pointers the caller has
 * pointed into dev_in, or anywhere else on the device -- and a copy of the B
 * sampled ids from args->out_idx (required) to host_out (host int64 [B],
 * pinned).  `sync` is one of FS_SYNC_*: FS_SYNC_STREAM waits for the stream;
 * FS_SYNC_IDS, when host_out is page-locked (the kernel then writes the ids
 * into it directly) and the stream had no pending work at the call (so no
 * earlier call can still write host_out), watches host_out until every id
 * has arrived, a few microseconds sooner than a stream wait (otherwise it
 * waits for the stream); FS_SYNC_NONE returns at once.  in_bytes may be 0 (inputs
 * already on the device).  Errors: FS_ERR_INVALID_ARG for a null args,
 * args->out_idx or host_out, a null host_in / dev_in with in_bytes > 0, or an
 * unknown sync; every error of fs_sample's argument checks -- all before
 * anything is enqueued; FS_ERR_CUDA for a failed copy, launch or wait (a watch
 * gives up after 10 s and reports the stream's status).
 */
fs_status fs_sample_host(const fs_sample_args *args, const void *host_in, void *dev_in,
                         size_t in_bytes, int64_t *host_out, int sync, void *stream);

/* Largest K of fs_sample_topk. */
#define FS_TOPK_MAX 16

/* Bytes of workspace fs_sample_topk needs: B * ceil(V/128) * C * 8 with
 * C = 4 for K <= 4 and 16 otherwise, rounded up to 256 (0 for bad sizes).
 * It needs no initialisation. */
size_t fs_topk_workspace_size(int64_t B, int64_t V, int64_t K);

/*
 * K distinct samples per row, without replacement, in draw order: the ids of
 * the K largest noisy scores s[b, v] (ties to the lower id).  By the Gumbel-
 * top-k property of the Gumbel-max trick this is a draw of K tokens without
 * replacement from softmax(l'[b, :]) (the aitrends.kr write-up notes the design
 * extends to top-k); out_topk_idx[b, 0] is the id fs_sample returns for the
 * same inputs.  Greedy rows give the K largest logits.  The stage-1 kernel
 * writes candidate lists -- the best 4 (K <= 4) or 16 (K <= 16) scores of each
 * run of tiles one thread saw of a row, in one (row, 128-id tile) slot of the
 * workspace, the run's other slots left empty -- to args->workspace
 * (fs_topk_workspace_size bytes, 256-byte aligned, no initialisation needed),
 * and a second kernel merges them per row.
 * Uses args' inputs (H, W, temperature, mask, seeds, offset, vocab_offset);
 * args' outputs (out_idx, out_tile_*, out_max, out_lse) must be NULL.
 * out_topk_idx: int64 [B, K] (-1 past the row's unmasked count);
 * out_topk_score: fp32 [B, K] or NULL (the scores, -inf past the count).
 */
fs_status fs_sample_topk(const fs_sample_args *args, int64_t K, int64_t *out_topk_idx,
                         float *out_topk_score, void *stream);

/* Merge rules of fs_group_merge. */
#define FS_MERGE_EXACT 0        /* argmax_k m_k: the sample of the union       */
#define FS_MERGE_GROUP_GUMBEL 1 /* argmax_k L_k + G_k with fresh Gumbel noise  */

/*
 * Combine per-partition results into one sample per row (aitrends.kr
 * write-up, tensor-parallel and Group-Gumbel-Max paragraphs; tomesphere
 * abstract: exact because argmax decomposes over partitions, grouped variants
 * exact by hierarchical factorisation).  Inputs are [P, B] row-major (the
 * partition's outputs one after another): z (int64 sampled global ids, -1 for
 * a fully masked row), m (fp32 maxima, for FS_MERGE_EXACT), L (fp32
 * log-masses, for FS_MERGE_GROUP_GUMBEL).
 *   FS_MERGE_EXACT:        out_idx[b] = z[k*, b], k* = argmax_k m[k, b] (lowest
 *                          k on ties); equals the unsharded sample when the
 *                          partitions were sampled with matching vocab_offset,
 *                          seeds and offset.
 *   FS_MERGE_GROUP_GUMBEL: k* = argmax_k (L[k, b] + G[k, b]), G Gumbel noise
 *                          independent of the partitions' own (Philox with the
 *                          row's seed, counter (k >> 2, b | 2^31, offset low,
 *                          offset high), word k & 3); out_idx[b] = z[k*, b].
 * Partitions with z < 0 or L = -inf are skipped; a row with none left gives -1.
 * out_L (optional, fp32 [B]) = log sum_k exp(L[k, b]) (needs L).  seeds: uint64
 * [B] or NULL for `seed`.  Device pointers; asynchronous on `stream`.
 */
fs_status fs_group_merge(const int64_t *z, const float *m, const float *L, int64_t P,
                         int64_t B, int mode, const uint64_t *seeds, uint64_t seed,
                         uint64_t offset, int64_t *out_idx, float *out_L, void *stream);

/*
 * The online form of the Group-Gumbel-Max merge (aitrends.kr write-up: binary
 * merge rule with O(1) state): fold the group `step` (new_z, new_L, [B]) into
 * the running state (state_z, state_L, [B], updated in place; start from
 * z = -1, L = -inf):  L' = logaddexp(L, new_L); with probability
 * exp(new_L - L') the state's sample becomes new_z; L <- L'.  The Bernoulli
 * uniform is the one fs_group_merge uses for partition k = step.  Groups with
 * new_z < 0 or new_L = -inf leave the state unchanged.
 */
fs_status fs_online_merge(int64_t *state_z, float *state_L, const int64_t *new_z,
                          const float *new_L, int64_t B, uint64_t step,
                          const uint64_t *seeds, uint64_t seed, uint64_t offset,
                          void *stream);

/*
 * Diagnostic: the Gumbel noise g[b, v] the stage-1 kernel adds, for rows
 * [b0, b0+nb) x ids [v0, v0+nv), written to out (device fp32 [nb, nv]).
 * seeds (device uint64 [b0+nb]) or NULL for `seed` on every row.  Same
 * Philox/uniform/log chain and the same device code as fs_sample
 * (aitrends.kr write-up, "Stage 1": g = -log(-log u)).
 */
fs_status fs_gumbel_noise(const uint64_t *seeds, uint64_t seed, uint64_t offset,
                          int64_t b0, int64_t nb, int64_t v0, int64_t nv,
                          float *out, void *stream);

/*
 * Diagnostic: the transform from one 32-bit Philox output word to the Gumbel
 * noise g the stage-1 kernel uses (the word's low 23 bits give
 * u = (k + 1/2) 2^-23, then g = -log(-log u)), applied to n given words
 * (device uint32 [n]) into out (device fp32 [n]) -- the same device code as
 * fs_sample, so every uniform level can be checked.  FS_ERR_INVALID_ARG for
 * n < 0 or null buffers with n > 0.
 */
fs_status fs_gumbel_transform(const uint32_t *words, int64_t n, float *out, void *stream);

/*
 * Diagnostic: run the sampling kernels' bounded wait on a barrier that nothing
 * ever arrives on, giving up after limit_ns (1e3 <= limit_ns <= 1e9).  The
 * kernel records the timeout in the device error word and returns, exactly as
 * a stalled sampling pipeline would, so a caller can check that timeouts are
 * reported (fs_last_device_error) and that the context stays usable, without
 * faulting or hanging the GPU.  FS_ERR_INVALID_ARG for a limit out of range.
 */
fs_status fs_wait_timeout_selftest(uint64_t limit_ns, void *stream);

/*
 * Read and clear the device-side error word of the current device, after the
 * work enqueued on `stream` so far (a cudaStream_t; NULL = the legacy default
 * stream): the read is a one-thread kernel and a copy on that stream, and the
 * call waits for that stream only.  *code receives the raw word (0 = none;
 * bit 0: a bounded pipeline wait timed out).  Returns FS_ERR_DEVICE_TIMEOUT if
 * a wait timed out since the last read, FS_OK otherwise, FS_ERR_CUDA on a
 * failed launch, copy or wait.
 * Scope: the word is one per device, not per stream or per call: every
 * sampling kernel on the device records its timeouts in it, so a timeout in a
 * call on another stream (or by another caller) is reported to whichever call
 * of this function reads it first, and one that is still running when this
 * call reads is reported by a later read.  A timeout means a pipeline wait
 * went 2 s without progress -- the device is in trouble for every caller --
 * so one report per device is what the word is for.  Two calls of this
 * function on one device at the same time share one snapshot word; serialise
 * them.
 */
fs_status fs_last_device_error(void *stream, int *code);

/* Human-readable name of a status code (static storage). */
const char *fs_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FS_SAMPLE_H_ */
