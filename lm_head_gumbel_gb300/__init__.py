"""Fused LM-head + exact Gumbel-max sampling (FlashSampling) for GB300.

The compute path is the C-ABI library ``libfs.so`` (CUDA, sm_103a); this
package is its Python binding plus the seeded synthetic workloads used by the
tests and the benchmark.
"""
from ._binding import (FS_ERR_CUDA, FS_ERR_DEVICE_TIMEOUT, FS_ERR_INVALID_ARG,  # noqa: F401
                       FS_ERR_UNSUPPORTED, FS_ERR_WORKSPACE, FS_FLAG_OVERLAP_PREVIOUS, FS_MERGE_EXACT,
                       FS_MERGE_GROUP_GUMBEL, FS_OK, FS_SYNC_IDS, FS_SYNC_NONE, FS_SYNC_STREAM,
                       FS_TILE, FS_TOPK_MAX, LIB_PATH, FsError,
                       FsSampleArgs, fs_group_merge, fs_gumbel_noise, fs_gumbel_transform,
                       fs_last_device_error,
                       fs_online_merge, fs_sample_topk, fs_topk_workspace_size,
                       fs_num_tiles, fs_sample, fs_sample_host, fs_status_string,
                       fs_wait_timeout_selftest,
                       fs_workspace_size,
                       load_library)
