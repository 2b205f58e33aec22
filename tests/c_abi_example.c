/*
 * The C ABI used from C alone (no Python, no PyTorch): device buffers from the
 * CUDA runtime, one greedy and one sampling call of fs_sample, the host-memory
 * step fs_sample_host, and argument errors.  Greedy rows (T = 0) must return
 * the argmax of the logits, which this program computes itself in double
 * precision from the same bf16 values (rows whose top-2 logits are closer than
 * 1e-3 are not judged); a call with FS_FLAG_OVERLAP_PREVIOUS must repeat the
 * plain call's ids; three draws without replacement on greedy rows must be the
 * three largest logits; two vocabulary shards merged exactly must give the
 * unsharded sample.  Prints "ok" and exits 0 on success.
 *
 * Built and run by tests/test_gpu_c_abi.py.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fs_sample.h"

#define CHECK(cond, msg)                                      \
  do {                                                        \
    if (!(cond)) {                                            \
      fprintf(stderr, "FAIL %s (line %d)\n", msg, __LINE__);  \
      return 1;                                               \
    }                                                         \
  } while (0)

/* float -> bf16 bits, round to nearest even (inputs are finite). */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* A small linear congruential stream mapped to roughly N(0, 1) (sum of 4). */
static uint64_t g_state = 12345;
static float next_normal(void) {
  float s = 0.0f;
  for (int i = 0; i < 4; ++i) {
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    s += (float)((g_state >> 40) & 0xFFFFFF) / 16777216.0f - 0.5f;
  }
  return s * 1.7320508f;
}

int main(void) {
  const int64_t B = 5, d = 64, V = 3000;
  const size_t nh = (size_t)(B * d), nw = (size_t)(V * d);
  uint16_t* hH = (uint16_t*)malloc(nh * 2);
  uint16_t* hW = (uint16_t*)malloc(nw * 2);
  for (size_t i = 0; i < nh; ++i) hH[i] = to_bf16(next_normal());
  for (size_t i = 0; i < nw; ++i) hW[i] = to_bf16(next_normal() * 0.25f);

  void *dH, *dW, *dT, *dws;
  int64_t* dout;
  CHECK(cudaMalloc(&dH, nh * 2) == cudaSuccess, "cudaMalloc H");
  CHECK(cudaMalloc(&dW, nw * 2) == cudaSuccess, "cudaMalloc W");
  CHECK(cudaMalloc(&dT, B * sizeof(float)) == cudaSuccess, "cudaMalloc T");
  CHECK(cudaMalloc((void**)&dout, B * sizeof(int64_t)) == cudaSuccess, "cudaMalloc out");
  const size_t ws_bytes = fs_workspace_size(B, V);
  CHECK(ws_bytes > 0, "fs_workspace_size");
  CHECK(cudaMalloc(&dws, ws_bytes) == cudaSuccess, "cudaMalloc workspace");
  CHECK(cudaMemset(dws, 0, ws_bytes) == cudaSuccess, "clear workspace");
  CHECK(cudaMemcpy(dH, hH, nh * 2, cudaMemcpyHostToDevice) == cudaSuccess, "copy H");
  CHECK(cudaMemcpy(dW, hW, nw * 2, cudaMemcpyHostToDevice) == cudaSuccess, "copy W");

  /* Greedy: T = 0 on every row. */
  float hT[5] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  CHECK(cudaMemcpy(dT, hT, sizeof hT, cudaMemcpyHostToDevice) == cudaSuccess, "copy T");
  fs_sample_args a;
  memset(&a, 0, sizeof a);
  a.H = dH;
  a.W = dW;
  a.temperature = (const float*)dT;
  a.seed = 7;
  a.offset = 0;
  a.B = B;
  a.d = d;
  a.V = V;
  a.ldh = d;
  a.ldw = d;
  a.out_idx = dout;
  a.workspace = dws;
  a.workspace_bytes = ws_bytes;
  CHECK(fs_sample(&a, NULL) == FS_OK, "fs_sample greedy");
  int64_t ids[5];
  CHECK(cudaMemcpy(ids, dout, sizeof ids, cudaMemcpyDeviceToHost) == cudaSuccess, "copy ids");
  int judged = 0;
  for (int64_t b = 0; b < B; ++b) {
    double best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int64_t v = 0; v < V; ++v) {
      double l = 0.0;
      for (int64_t k = 0; k < d; ++k) l += from_bf16(hH[b * d + k]) * from_bf16(hW[v * d + k]);
      if (l > best) {
        second = best;
        best = l;
        arg = v;
      } else if (l > second) {
        second = l;
      }
    }
    if (best - second > 1e-3) {
      CHECK(ids[b] == arg, "greedy id is the argmax");
      ++judged;
    }
  }
  CHECK(judged >= 3, "enough clearly separated rows");

  /* Sampling (T = 1): ids in range and the same on a repeated call. */
  for (int64_t b = 0; b < B; ++b) hT[b] = 1.0f;
  CHECK(cudaMemcpy(dT, hT, sizeof hT, cudaMemcpyHostToDevice) == cudaSuccess, "copy T");
  a.offset = 11;
  CHECK(fs_sample(&a, NULL) == FS_OK, "fs_sample T=1");
  int64_t first[5], again[5];
  CHECK(cudaMemcpy(first, dout, sizeof first, cudaMemcpyDeviceToHost) == cudaSuccess, "copy");
  for (int64_t b = 0; b < B; ++b) CHECK(first[b] >= 0 && first[b] < V, "id in range");

  /* The same call launched to overlap the kernel before it: the same ids. */
  a.flags = FS_FLAG_OVERLAP_PREVIOUS;
  CHECK(fs_sample(&a, NULL) == FS_OK, "fs_sample T=1 overlapped");
  CHECK(cudaMemcpy(again, dout, sizeof again, cudaMemcpyDeviceToHost) == cudaSuccess, "copy");
  for (int64_t b = 0; b < B; ++b) CHECK(again[b] == first[b], "overlapped call = plain call");
  a.flags = 0;

  /* The same call from host memory: H and T copied in, ids written back. */
  const size_t in_bytes = nh * 2 + 256;
  void* host_in = NULL;
  int64_t* host_out = NULL;
  void* dev_in = NULL;
  CHECK(cudaMallocHost(&host_in, in_bytes) == cudaSuccess, "pinned in");
  CHECK(cudaMallocHost((void**)&host_out, B * sizeof(int64_t)) == cudaSuccess, "pinned out");
  CHECK(cudaMalloc(&dev_in, in_bytes) == cudaSuccess, "dev_in");
  memcpy(host_in, hH, nh * 2);
  memcpy((char*)host_in + nh * 2, hT, sizeof hT);
  fs_sample_args h = a;
  h.H = dev_in;
  h.temperature = (const float*)((char*)dev_in + nh * 2);
  CHECK(fs_sample_host(&h, host_in, dev_in, in_bytes, host_out, 1, NULL) == FS_OK,
        "fs_sample_host");
  for (int64_t b = 0; b < B; ++b) again[b] = host_out[b];
  for (int64_t b = 0; b < B; ++b) CHECK(again[b] == first[b], "host step = device call");

  /* K draws without replacement, greedy rows: the K largest logits in order.
   * Each row's three largest logits are found here in double precision; rows
   * whose top logits are closer than 1e-3 are not judged. */
  for (int64_t b = 0; b < B; ++b) hT[b] = 0.0f;
  CHECK(cudaMemcpy(dT, hT, sizeof hT, cudaMemcpyHostToDevice) == cudaSuccess, "copy T");
  {
    const int64_t K = 3;
    void* tk_ws = NULL;
    int64_t* tk_out = NULL;
    const size_t tk_bytes = fs_topk_workspace_size(B, V, K);
    CHECK(tk_bytes > 0, "fs_topk_workspace_size");
    CHECK(cudaMalloc(&tk_ws, tk_bytes) == cudaSuccess, "cudaMalloc top-K workspace");
    CHECK(cudaMalloc((void**)&tk_out, B * K * sizeof(int64_t)) == cudaSuccess, "cudaMalloc top-K");
    fs_sample_args t = a;
    t.out_idx = NULL;
    t.workspace = tk_ws;
    t.workspace_bytes = tk_bytes;
    CHECK(fs_sample_topk(&t, K, tk_out, NULL, NULL) == FS_OK, "fs_sample_topk");
    int64_t got[5 * 3];
    CHECK(cudaMemcpy(got, tk_out, sizeof got, cudaMemcpyDeviceToHost) == cudaSuccess, "copy");
    int judged_k = 0;
    for (int64_t b = 0; b < B; ++b) {
      double top[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      int64_t arg[4] = {-1, -1, -1, -1};
      for (int64_t v = 0; v < V; ++v) {
        double l = 0.0;
        for (int64_t k = 0; k < d; ++k) l += from_bf16(hH[b * d + k]) * from_bf16(hW[v * d + k]);
        int q = 4;
        while (q > 0 && l > top[q - 1]) --q;
        if (q < 4) {
          for (int r = 3; r > q; --r) {
            top[r] = top[r - 1];
            arg[r] = arg[r - 1];
          }
          top[q] = l;
          arg[q] = v;
        }
      }
      if (top[0] - top[1] > 1e-3 && top[1] - top[2] > 1e-3 && top[2] - top[3] > 1e-3) {
        for (int q = 0; q < 3; ++q) CHECK(got[b * K + q] == arg[q], "top-K id is the q-th logit");
        ++judged_k;
      }
    }
    CHECK(judged_k >= 2, "enough clearly separated rows for top-K");
    cudaFree(tk_ws);
    cudaFree(tk_out);
  }

  /* Two vocabulary shards sampled with global ids, merged exactly: the same
   * ids as the unsharded call (T = 1, the offset of `first`). */
  for (int64_t b = 0; b < B; ++b) hT[b] = 1.0f;
  CHECK(cudaMemcpy(dT, hT, sizeof hT, cudaMemcpyHostToDevice) == cudaSuccess, "copy T");
  {
    const int64_t cut = 1536; /* a multiple of 256: the shards keep the unsharded K order */
    int64_t* z = NULL;
    float* m = NULL;
    int64_t* merged = NULL;
    CHECK(cudaMalloc((void**)&z, 2 * B * sizeof(int64_t)) == cudaSuccess, "cudaMalloc z");
    CHECK(cudaMalloc((void**)&m, 2 * B * sizeof(float)) == cudaSuccess, "cudaMalloc m");
    CHECK(cudaMalloc((void**)&merged, B * sizeof(int64_t)) == cudaSuccess, "cudaMalloc merged");
    for (int part = 0; part < 2; ++part) {
      fs_sample_args s = a;
      s.offset = 11;
      s.W = (const char*)dW + (part ? cut * d * 2 : 0);
      s.V = part ? V - cut : cut;
      s.vocab_offset = part ? cut : 0;
      s.out_idx = z + part * B;
      s.out_max = m + part * B;
      CHECK(fs_sample(&s, NULL) == FS_OK, "fs_sample on a shard");
    }
    CHECK(fs_group_merge(z, m, NULL, 2, B, FS_MERGE_EXACT, NULL, 7, 11, merged, NULL, NULL) ==
              FS_OK,
          "fs_group_merge");
    int64_t mg[5];
    CHECK(cudaMemcpy(mg, merged, sizeof mg, cudaMemcpyDeviceToHost) == cudaSuccess, "copy");
    for (int64_t b = 0; b < B; ++b) CHECK(mg[b] == first[b], "merged shards = unsharded sample");
    cudaFree(z);
    cudaFree(m);
    cudaFree(merged);
  }

  /* Errors come back as status codes, before anything runs. */
  fs_sample_args bad = a;
  bad.B = 0;
  CHECK(fs_sample(&bad, NULL) == FS_ERR_INVALID_ARG, "B = 0 rejected");
  bad = a;
  bad.workspace = NULL;
  CHECK(fs_sample(&bad, NULL) == FS_ERR_WORKSPACE, "missing workspace rejected");
  CHECK(strcmp(fs_status_string(FS_ERR_WORKSPACE), "FS_ERR_WORKSPACE") == 0, "status string");
  int code = -1;
  CHECK(fs_last_device_error(NULL, &code) == FS_OK && code == 0, "no device error");

  cudaFreeHost(host_in);
  cudaFreeHost(host_out);
  cudaFree(dev_in);
  cudaFree(dH);
  cudaFree(dW);
  cudaFree(dT);
  cudaFree(dout);
  cudaFree(dws);
  free(hH);
  free(hW);
  printf("ok\n");
  return 0;
}
