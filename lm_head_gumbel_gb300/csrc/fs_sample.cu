// fs_sample.cu -- host side of the fused LM-head + exact Gumbel-max sampler:
// argument checks, TMA tensor maps, launch configuration, and the C ABI
// declared in fs_sample.h.  The kernels are in fs_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <chrono>
#include <climits>
#include <mutex>

#include "fs_kernels.cuh"
#include "fs_sample.h"

namespace fs {

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr int kNumModes = 4;
struct DeviceState {
  bool initialised = false;
  fs_status status = FS_ERR_UNSUPPORTED;
  int num_sms = 0;
  int max_pairs[kNumModes] = {};  // co-resident CTA pairs of the pair kernel, per mode
};

std::mutex g_mu;
DeviceState g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
thread_local const DeviceState* g_last_state = nullptr;  // set by device_setup
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// attr must hold two entries: the cluster shape (cluster > 1) and, with pdl,
// programmatic stream serialization (the kernel may start before the previous
// one on the stream ends; it resolves the dependency itself).
cudaLaunchConfig_t launch_config(int cluster, cudaLaunchAttribute* attr, cudaStream_t stream,
                                 size_t smem, bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  unsigned n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = unsigned(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

// Opt both stage-1 kernels of one epilogue mode into their shared memory and
// record how many CTA pairs fit on the device at once (the pair kernel's
// persistent grid).
template <int kMode>
bool prepare_mode(DeviceState& st, int sms) {
  if (cudaFuncSetAttribute(stage1_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes)) != cudaSuccess)
    return false;
  auto pk = stage1_pair_kernel<kMode, false>;
  if (cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kPairSmemBytes)) != cudaSuccess)
    return false;
  if constexpr (kTopkMode<kMode>) {  // the grouped unit order (same resources)
    if (cudaFuncSetAttribute(stage1_pair_kernel<kMode, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPairSmemBytes)) != cudaSuccess)
      return false;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(2, attr, nullptr, kPairSmemBytes);
  cfg.gridDim = dim3(unsigned((sms / 2) * 2), 1, 1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, pk, &cfg) != cudaSuccess || n < 1) return false;
  st.max_pairs[kMode] = n;
  return true;
}

// Persistent grid size for n_units units on at most `slots` co-resident CTAs
// (or CTA pairs): the smallest grid that still needs no more waves than the
// full one.  Every CTA then takes its units in the same number of rounds, so
// no thin last wave streams W with a fraction of the SMs (the Llama-3 head's
// 501 units on 152 SMs: 126 CTAs of 4 units instead of 3.3 waves, 6-7 %
// faster); when the last wave is nearly full it changes nothing.
int balanced_grid(int n_units, int slots) {
  if (n_units <= slots) return n_units;
  const int waves = (n_units + slots - 1) / slots;
  return (n_units + waves - 1) / waves;
}

template <int kMode>
fs_status launch_mode(bool pair, const CUtensorMap& tmap_h, const CUtensorMap& tmap_w,
                      const Stage1Params& p, const DeviceState& ds, cudaStream_t stream) {
  const int n_vt = int((int64_t(p.V) + kBlockN - 1) / kBlockN);
  cudaLaunchAttribute attr[2];
  cudaError_t err;
  if (pair) {
    const int n_mp = int((int64_t(p.B) + 2 * kBlockM - 1) / (2 * kBlockM));
    const int n_units = n_vt * n_mp;
    const int pairs = balanced_grid(n_units, ds.max_pairs[kMode]);
    // The top-K modes' grouped unit order (pair_unit in fs_kernels.cuh) when
    // it needs no more waves than the plain one: groups of n_mp pairs walk
    // `waves` vocabulary blocks each, and the pairs left over take the rest.
    Stage1Params q = p;
    if (kTopkMode<kMode> && n_mp > 1) {
      const int waves = (n_units + pairs - 1) / pairs;
      const int groups = pairs / n_mp, n_left = pairs - groups * n_mp;
      const int left = n_vt - std::min(n_vt, groups * waves);
      if (groups > 0 &&
          (left == 0 || (n_left > 0 && ((left + n_left - 1) / n_left) * n_mp <= waves))) {
        q.pair_groups = groups;
        q.pair_group_blocks = waves;
      }
    }
    cudaLaunchConfig_t cfg = launch_config(2, attr, stream, kPairSmemBytes, p.pdl != 0);
    cfg.gridDim = dim3(unsigned(pairs * 2), 1, 1);
    if constexpr (kTopkMode<kMode>) {
      if (q.pair_groups > 0)
        err = cudaLaunchKernelEx(&cfg, stage1_pair_kernel<kMode, true>, tmap_h, tmap_w, q);
      else
        err = cudaLaunchKernelEx(&cfg, stage1_pair_kernel<kMode, false>, tmap_h, tmap_w, q);
    } else {
      err = cudaLaunchKernelEx(&cfg, stage1_pair_kernel<kMode, false>, tmap_h, tmap_w, q);
    }
  } else {
    const int n_units = n_vt * p.n_mt;
    const int grid = balanced_grid(n_units, ds.num_sms);
    cudaLaunchConfig_t cfg = launch_config(1, attr, stream, kSmemBytes, p.pdl != 0);
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    err = cudaLaunchKernelEx(&cfg, stage1_kernel<kMode>, tmap_h, tmap_w, p);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return FS_ERR_CUDA;
  }
  return FS_OK;
}

fs_status device_setup(int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FS_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_devices[dev];
  if (!st.initialised) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FS_ERR_CUDA;
    }
    st.num_sms = sms;
    if (major != 10 || minor != 3) {
      st.status = FS_ERR_UNSUPPORTED;
    } else {
      st.status = FS_OK;
      if (!prepare_mode<kModeSample>(st, sms) || !prepare_mode<kModeLse>(st, sms) ||
          !prepare_mode<kModeTop4>(st, sms) || !prepare_mode<kModeTop16>(st, sms)) {
        cudaGetLastError();
        st.status = FS_ERR_CUDA;
      }
      if (st.status == FS_OK && g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          st.status = FS_ERR_CUDA;
        } else {
          g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
      }
    }
    st.initialised = true;
  }
  *num_sms = st.num_sms;
  g_last_state = &st;
  return st.status;
}

// 2-D bf16 tensor map: inner extent `inner` (contiguous), `outer` rows of
// `row_bytes`; boxes of box_inner x box_outer with the 128-byte swizzle;
// out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace fs

using namespace fs;

// Defined in fs_merge.cu: the per-row log-sum-exp over the tile log-masses.
namespace fs {
fs_status launch_row_lse(const float* tile_lse, const float* temperature, int64_t B,
                         int64_t n_tiles, float* out_lse, cudaStream_t stream);
// Defined in fs_merge.cu: each row's K best of its per-tile top-K candidates.
fs_status launch_topk_reduce(const float* cand_score, const int32_t* cand_idx, int64_t B,
                             int64_t n_tiles, int64_t cap, int64_t K, int64_t* out_idx,
                             float* out_score, cudaStream_t stream);
}

extern "C" int64_t fs_num_tiles(int64_t V) { return V <= 0 ? 0 : (V + kTileV - 1) / kTileV; }

// Workspace layout: [0, 4) the CTA ticket, [256, 256 + 8B) the per-row keys.
constexpr size_t kKeysOffset = 256;

extern "C" size_t fs_workspace_size(int64_t B, int64_t V) {
  if (B <= 0 || V <= 0) return 0;
  const size_t bytes = kKeysOffset + size_t(B) * 8u;
  return (bytes + 255u) & ~size_t(255u);
}

extern "C" const char* fs_status_string(int status) {
  switch (status) {
    case FS_OK: return "FS_OK";
    case FS_ERR_INVALID_ARG: return "FS_ERR_INVALID_ARG";
    case FS_ERR_UNSUPPORTED: return "FS_ERR_UNSUPPORTED";
    case FS_ERR_CUDA: return "FS_ERR_CUDA";
    case FS_ERR_DEVICE_TIMEOUT: return "FS_ERR_DEVICE_TIMEOUT";
    case FS_ERR_WORKSPACE: return "FS_ERR_WORKSPACE";
    default: return "FS_ERR_UNKNOWN";
  }
}

namespace fs {
namespace {

// Checks shared by every sampling entry point: the inputs of fs_sample_args.
fs_status check_inputs(const fs_sample_args* a) {
  if (a == nullptr) return FS_ERR_INVALID_ARG;
  const int64_t B = a->B, d = a->d, V = a->V;
  if (!a->H || !a->W) return FS_ERR_INVALID_ARG;
  if ((a->flags & ~uint32_t(FS_FLAG_OVERLAP_PREVIOUS)) != 0) return FS_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || d < 1 || V < 1 || V > int64_t(0x7FFFFFFF)) return FS_ERR_INVALID_ARG;
  if (d > int64_t(0x7FFFFFFF) - kBlockK) return FS_ERR_INVALID_ARG;
  if (a->ldh < d || a->ldw < d || a->ldh % 8 != 0 || a->ldw % 8 != 0) return FS_ERR_INVALID_ARG;
  if (!aligned(a->H, 16) || !aligned(a->W, 16)) return FS_ERR_INVALID_ARG;
  if (a->temperature && !aligned(a->temperature, 4)) return FS_ERR_INVALID_ARG;
  if (a->seeds && !aligned(a->seeds, 8)) return FS_ERR_INVALID_ARG;
  if (a->vocab_mask && (!aligned(a->vocab_mask, 4) || a->mask_ld < (V + 31) / 32))
    return FS_ERR_INVALID_ARG;
  if (a->vocab_offset < 0 || a->vocab_offset % 4 != 0 ||
      a->vocab_offset + V > int64_t(0x7FFFFFFF))
    return FS_ERR_INVALID_ARG;
  // The kernels count work units ((V / 256) x (B / 128)) in 32-bit integers.
  if (((V + kBlockN - 1) / kBlockN) * ((B + kBlockM - 1) / kBlockM) > int64_t(0x7FFFFFFF))
    return FS_ERR_INVALID_ARG;
  return FS_OK;
}

// Encode the tensor maps, fill the kernel parameters and launch the stage-1
// kernel of `mode` (single CTAs, or CTA pairs for an even number of 128-row
// batch blocks).  `p` arrives with the output pointers set.
fs_status run_stage1(const fs_sample_args* a, int mode, Stage1Params& p, cudaStream_t stream,
                     bool pdl = false) {
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  const int64_t B = a->B, d = a->d, V = a->V;
  // H box: only the rows that exist (rounded up to the 8-row swizzle atom);
  // the MMA's remaining A rows hold stale data and only feed accumulator rows
  // that are never read.
  const uint32_t h_rows = B >= kBlockM ? uint32_t(kBlockM) : uint32_t((B + 7) / 8 * 8);
  const int n_mt = int((B + kBlockM - 1) / kBlockM);
  // An even number of 128-row batch blocks: CTA pairs with M = 256 MMAs, each
  // CTA holding half of the W slice (six 32 KB stages).  Otherwise single
  // CTAs with M = 128 and the whole slice (4-5 stages of H box + 32 KB); with
  // an odd number of batch blocks above one, pairs would leave half a pair idle.
  const bool pair = n_mt > 1 && n_mt % 2 == 0;
  CUtensorMap tmap_h, tmap_w;
  if (!encode_2d(&tmap_h, a->H, uint64_t(d), uint64_t(B), uint64_t(a->ldh) * 2u, kBlockK,
                 h_rows) ||
      !encode_2d(&tmap_w, a->W, uint64_t(d), uint64_t(V), uint64_t(a->ldw) * 2u, kBlockK,
                 uint32_t(pair ? kBlockN / 2 : kBlockN)))
    return FS_ERR_INVALID_ARG;
  p.B = int32_t(B);
  p.V = int32_t(V);
  p.n_tiles = int32_t(fs_num_tiles(V));
  p.n_mt = int32_t(n_mt);
  p.n_kb = int32_t((d + kBlockK - 1) / kBlockK);
  p.temperature = a->temperature;
  p.mask = a->vocab_mask;
  p.mask_ld = a->mask_ld;
  p.seeds = a->seeds;
  p.seed = a->seed;
  p.offset = a->offset;
  p.vocab_offset = int32_t(a->vocab_offset);
  p.wait_limit_ns = kWaitLimitNs;
  p.h_box_rows = h_rows;
  p.pdl = pdl ? 1u : 0u;
  p.stage_bytes = h_rows * 128u + kSmemB;  // h_rows is a multiple of 8: 1 KB swizzle atoms
  p.n_stages = kRingBytes / p.stage_bytes < uint32_t(kMaxStages) ? kRingBytes / p.stage_bytes
                                                                : uint32_t(kMaxStages);
  const DeviceState& ds = *g_last_state;
  switch (mode) {
    case kModeSample: return launch_mode<kModeSample>(pair, tmap_h, tmap_w, p, ds, stream);
    case kModeLse: return launch_mode<kModeLse>(pair, tmap_h, tmap_w, p, ds, stream);
    case kModeTop4: return launch_mode<kModeTop4>(pair, tmap_h, tmap_w, p, ds, stream);
    default: return launch_mode<kModeTop16>(pair, tmap_h, tmap_w, p, ds, stream);
  }
}

}  // namespace
}  // namespace fs

namespace fs {
namespace {
// Every host-side check of fs_sample (inputs, outputs, workspace).
fs_status check_sample(const fs_sample_args* a) {
  const fs_status chk = check_inputs(a);
  if (chk != FS_OK) return chk;
  const int64_t B = a->B, V = a->V;
  if (!a->out_idx && !a->out_tile_max) return FS_ERR_INVALID_ARG;
  if (a->out_idx && !aligned(a->out_idx, 8)) return FS_ERR_INVALID_ARG;
  if ((a->out_tile_max == nullptr) != (a->out_tile_idx == nullptr)) return FS_ERR_INVALID_ARG;
  if (a->out_tile_max && (!aligned(a->out_tile_max, 4) || !aligned(a->out_tile_idx, 4)))
    return FS_ERR_INVALID_ARG;
  if (a->out_tile_lse && (!aligned(a->out_tile_lse, 4) || !a->out_tile_max))
    return FS_ERR_INVALID_ARG;
  if (a->out_max && (!a->out_idx || !aligned(a->out_max, 4))) return FS_ERR_INVALID_ARG;
  if (a->out_lse && (!a->out_tile_lse || !aligned(a->out_lse, 4))) return FS_ERR_INVALID_ARG;
  if (a->out_idx != nullptr) {
    const size_t need = fs_workspace_size(B, V);
    if (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 256))
      return FS_ERR_WORKSPACE;
  }
  return FS_OK;
}
}  // namespace
}  // namespace fs

namespace fs {
namespace {
// fs_sample, optionally also writing the ids to `out_idx_host` (a device
// address of mapped host memory); with pdl the kernel overlaps the kernel
// before it on the stream, which writes its H and per-row inputs.
fs_status sample(const fs_sample_args* a, int64_t* out_idx_host, bool pdl, void* stream_ptr) {
  const fs_status chk = check_sample(a);
  if (chk != FS_OK) return chk;
  const int64_t B = a->B, V = a->V;
  Stage1Params p = {};
  p.tile_max = a->out_tile_max;
  p.tile_idx = a->out_tile_idx;
  p.tile_lse = a->out_tile_lse;
  p.out_idx = a->out_idx;
  p.out_idx_host = out_idx_host;
  p.out_max = a->out_max;
  p.ticket = a->out_idx ? static_cast<uint32_t*>(a->workspace) : nullptr;
  p.row_keys = a->out_idx ? reinterpret_cast<unsigned long long*>(
                                static_cast<uint8_t*>(a->workspace) + kKeysOffset)
                          : nullptr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const fs_status lst = run_stage1(a, a->out_tile_lse ? kModeLse : kModeSample, p, stream, pdl);
  if (lst != FS_OK || a->out_lse == nullptr) return lst;
  return launch_row_lse(a->out_tile_lse, a->temperature, B, fs_num_tiles(V), a->out_lse, stream);
}

// Device address of host memory the GPU can read and write directly (pinned
// and mapped, as page-locked allocations are under unified addressing), or
// null if `host` is not such memory.
void* mapped_host(const void* host) {
  cudaPointerAttributes at = {};
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

constexpr int64_t kIdPending = INT64_MIN;

// Wait until every entry of the mapped host buffer `ids` has been written by
// the kernel (none is kIdPending any more).  Bounded: after 10 s of waiting,
// or if the stream reports an error, the stream's own status decides.
fs_status watch_ids(const int64_t* ids, int64_t n, cudaStream_t stream) {
  const volatile int64_t* v = ids;
  const auto t0 = std::chrono::steady_clock::now();
  for (int64_t b = 0; b < n; ++b) {
    while (v[b] == kIdPending) {
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10)) {
        const cudaError_t e = cudaStreamSynchronize(stream);
        cudaGetLastError();
        return e == cudaSuccess && v[b] != kIdPending ? FS_OK : FS_ERR_CUDA;
      }
    }
  }
  std::atomic_thread_fence(std::memory_order_acquire);
  return FS_OK;
}

// Whether W (the one input the overlapped kernel reads before the copy in is
// complete) lies in the buffer that copy writes.
bool w_in_buffer(const fs_sample_args* a, const void* buf, size_t bytes) {
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(a->W);
  const uintptr_t w1 = w0 + uintptr_t(a->V - 1) * uintptr_t(a->ldw) * 2u + uintptr_t(a->d) * 2u;
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(buf), b1 = b0 + bytes;
  return w0 < b1 && b0 < w1;
}
}  // namespace
}  // namespace fs

extern "C" fs_status fs_sample(const fs_sample_args* a, void* stream_ptr) {
  return sample(a, nullptr, a != nullptr && (a->flags & FS_FLAG_OVERLAP_PREVIOUS) != 0,
                stream_ptr);
}

extern "C" size_t fs_topk_workspace_size(int64_t B, int64_t V, int64_t K) {
  if (B <= 0 || V <= 0 || K < 1 || K > FS_TOPK_MAX) return 0;
  const size_t cap = K <= 4 ? 4u : 16u;
  const size_t bytes = size_t(B) * size_t(fs_num_tiles(V)) * cap * 8u;
  return (bytes + 255u) & ~size_t(255u);
}

extern "C" fs_status fs_sample_topk(const fs_sample_args* a, int64_t K, int64_t* out_topk_idx,
                                    float* out_topk_score, void* stream_ptr) {
  const fs_status chk = check_inputs(a);
  if (chk != FS_OK) return chk;
  const int64_t B = a->B, V = a->V;
  if (K < 1 || K > FS_TOPK_MAX || !out_topk_idx || !aligned(out_topk_idx, 8) ||
      (out_topk_score && !aligned(out_topk_score, 4)))
    return FS_ERR_INVALID_ARG;
  if (a->out_idx || a->out_tile_max || a->out_tile_idx || a->out_tile_lse || a->out_max ||
      a->out_lse)
    return FS_ERR_INVALID_ARG;
  const size_t need = fs_topk_workspace_size(B, V, K);
  if (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 256))
    return FS_ERR_WORKSPACE;
  const int cap = K <= 4 ? 4 : 16;
  const int64_t n_cand = fs_num_tiles(V) * cap;
  Stage1Params p = {};
  p.topk_score = static_cast<float*>(a->workspace);
  p.topk_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a->workspace) +
                                          size_t(B) * size_t(n_cand) * 4u);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const fs_status lst = run_stage1(a, cap == 4 ? kModeTop4 : kModeTop16, p, stream,
                                   (a->flags & FS_FLAG_OVERLAP_PREVIOUS) != 0);
  if (lst != FS_OK) return lst;
  return launch_topk_reduce(p.topk_score, p.topk_idx, B, fs_num_tiles(V), cap, K, out_topk_idx,
                            out_topk_score, stream);
}

// ---- allocation-free variant ---------------------------------------------
// Scratch of fs_sample_noalloc: a file-scope device array, so callers that
// cannot allocate device memory still have the per-row reduction workspace.
// In host code `g_noalloc_scratch` is only a host-side stand-in for the symbol;
// its device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FS_NOALLOC_SCRATCH_BYTES];

namespace fs {
namespace {
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call per device.  That call also clears the array with a memset
// enqueued on the caller's stream, so the sampling kernel that follows on the
// same stream sees it cleared whatever kind of stream it is (a plain
// cudaMemset would go to the legacy default stream, which a non-blocking
// stream does not wait for).
fs_status noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FS_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr ||
        cudaMemsetAsync(p, 0, FS_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess) {
      cudaGetLastError();
      return FS_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FS_OK;
}
}  // namespace
}  // namespace fs

extern "C" fs_status fs_sample_noalloc(const fs_sample_args* a, void* stream_ptr) {
  if (a == nullptr) return FS_ERR_INVALID_ARG;
  if (a->out_idx != nullptr) {  // the built-in scratch must hold the workspace
    if (a->B < 1 || a->B > 65535 || a->V < 1 || a->V > int64_t(0x7FFFFFFF))
      return FS_ERR_INVALID_ARG;
    if (fs_workspace_size(a->B, a->V) > FS_NOALLOC_SCRATCH_BYTES) return FS_ERR_WORKSPACE;
  }
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  void* scratch = nullptr;
  const fs_status st2 = noalloc_scratch(static_cast<cudaStream_t>(stream_ptr), &scratch);
  if (st2 != FS_OK) return st2;
  fs_sample_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = FS_NOALLOC_SCRATCH_BYTES;
  return fs_sample(&b, stream_ptr);
}

extern "C" fs_status fs_sample_host(const fs_sample_args* a, const void* host_in, void* dev_in,
                                    size_t in_bytes, int64_t* host_out, int sync,
                                    void* stream_ptr) {
  if (a == nullptr || host_out == nullptr || a->out_idx == nullptr) return FS_ERR_INVALID_ARG;
  if (sync != FS_SYNC_NONE && sync != FS_SYNC_STREAM && sync != FS_SYNC_IDS)
    return FS_ERR_INVALID_ARG;
  if (in_bytes > 0 && (host_in == nullptr || dev_in == nullptr)) return FS_ERR_INVALID_ARG;
  const fs_status chk = check_sample(a);
  if (chk != FS_OK) return chk;
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  // Ids out: the kernel's last CTA writes them to mapped host memory as well;
  // otherwise they are copied back.  Watching host_out for them is safe only
  // if nothing enqueued earlier on the stream (an earlier call that did not
  // wait) can still write it; otherwise the call waits for the stream.
  int64_t* out_mapped = static_cast<int64_t*>(mapped_host(host_out));
  bool watch = sync == FS_SYNC_IDS && out_mapped != nullptr;
  if (watch) {
    const cudaError_t q = cudaStreamQuery(stream);
    if (q != cudaSuccess) {
      if (q != cudaErrorNotReady) {
        cudaGetLastError();
        return FS_ERR_CUDA;
      }
      cudaGetLastError();
      watch = false;
    }
  }
  if (watch) {  // no id is ever this value, so each entry shows when it lands
    for (int64_t b = 0; b < a->B; ++b) host_out[b] = kIdPending;
  }
  // Inputs in: mapped host memory is read by SMs over the host link (on a
  // Grace host, NVLink-C2C: several times the copy engine's rate for a
  // decode-sized H); other host memory goes through cudaMemcpyAsync.
  // The sampling kernel overlaps the copy kernel below, or, with no inputs to
  // copy and the flag set, whatever kernel came before on the stream.
  bool overlap = in_bytes == 0 && (a->flags & FS_FLAG_OVERLAP_PREVIOUS) != 0;
  if (in_bytes > 0) {
    const void* src = mapped_host(host_in);
    if (src != nullptr) {
      overlap = !w_in_buffer(a, dev_in, in_bytes);
      const int vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(dev_in) % 16 == 0) ? 1 : 0;
      const size_t per_block = 256u * (vec ? 16u : 1u);
      size_t blocks = (in_bytes + per_block - 1) / per_block;
      if (blocks > size_t(num_sms) * 4u) blocks = size_t(num_sms) * 4u;
      stage_in_kernel<<<unsigned(blocks), 256, 0, stream>>>(
          static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dev_in), in_bytes, vec);
      if (cudaGetLastError() != cudaSuccess) return FS_ERR_CUDA;
    } else if (cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, stream) !=
               cudaSuccess) {
      cudaGetLastError();
      return FS_ERR_CUDA;
    }
  }
  const fs_status run = sample(a, out_mapped, overlap, stream_ptr);
  if (run != FS_OK) return run;
  if (out_mapped == nullptr &&
      cudaMemcpyAsync(host_out, a->out_idx, size_t(a->B) * sizeof(int64_t),
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess) {
    cudaGetLastError();
    return FS_ERR_CUDA;
  }
  if (watch) return watch_ids(host_out, a->B, stream);
  if (sync && cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return FS_ERR_CUDA;
  }
  return FS_OK;
}

extern "C" fs_status fs_gumbel_transform(const uint32_t* words, int64_t n, float* out,
                                         void* stream_ptr) {
  if (n < 0 || (n > 0 && (!words || !out))) return FS_ERR_INVALID_ARG;
  if (n == 0) return FS_OK;
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  if (blocks > int64_t(0x7FFFFFFF)) return FS_ERR_INVALID_ARG;
  gumbel_transform_kernel<<<unsigned(blocks), threads, 0, static_cast<cudaStream_t>(stream_ptr)>>>(
      words, n, out);
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

extern "C" fs_status fs_gumbel_noise(const uint64_t* seeds, uint64_t seed, uint64_t offset,
                                     int64_t b0, int64_t nb, int64_t v0, int64_t nv, float* out,
                                     void* stream_ptr) {
  if (!out || b0 < 0 || nb < 0 || v0 < 0 || nv < 0) return FS_ERR_INVALID_ARG;
  if (b0 + nb > int64_t(0xFFFFFFFF) || v0 + nv > int64_t(0x7FFFFFFF)) return FS_ERR_INVALID_ARG;
  if (nb == 0 || nv == 0) return FS_OK;
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  const int64_t n = nb * nv;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  if (blocks > int64_t(0x7FFFFFFF)) return FS_ERR_INVALID_ARG;
  noise_kernel<<<unsigned(blocks), threads, 0, static_cast<cudaStream_t>(stream_ptr)>>>(
      seeds, seed, offset, b0, nb, v0, nv, out);
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

extern "C" fs_status fs_wait_timeout_selftest(uint64_t limit_ns, void* stream_ptr) {
  if (limit_ns < 1000u || limit_ns > 1000000000u) return FS_ERR_INVALID_ARG;
  int num_sms = 0;
  const fs_status st = device_setup(&num_sms);
  if (st != FS_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream_ptr)>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

namespace fs {
// Take the device error word (read it and clear it in one atomic step) into
// g_error_taken, ordered on the stream of the caller that asks for it.
__device__ int g_error_taken = 0;
__global__ void take_error_word_kernel() { g_error_taken = atomicExch(&g_error_word, 0); }
}  // namespace fs

extern "C" fs_status fs_last_device_error(void* stream_ptr, int* code) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int v = 0;
  take_error_word_kernel<<<1, 1, 0, stream>>>();
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&v, g_error_taken, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return FS_ERR_CUDA;
  }
  if (code) *code = v;
  return (v & kErrWaitTimeout) ? FS_ERR_DEVICE_TIMEOUT : FS_OK;
}
