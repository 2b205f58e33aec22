"""Failure detection without a GPU fault: the sampling kernels' bounded wait,
run on a barrier that nothing arrives on, gives up after its limit, the
timeout is reported through fs_last_device_error (and cleared by reading it),
and the context keeps working."""
import numpy as np
import pytest
import torch

import lm_head_gumbel_gb300 as fs
from gpu_cases import compare, make_problem, run_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()


def test_wait_timeout_is_reported_and_cleared():
    assert fs.fs_last_device_error() == (fs.FS_OK, 0)
    fs.fs_wait_timeout_selftest(2_000_000)  # 2 ms
    st, code = fs.fs_last_device_error()
    assert st == fs.FS_ERR_DEVICE_TIMEOUT and code & 1
    assert fs.fs_last_device_error() == (fs.FS_OK, 0)


def test_context_usable_after_timeout():
    fs.fs_wait_timeout_selftest(1_000_000)
    p = make_problem(8, 128, 2000, T=1.0, seed=21)
    dev = run_device(p, offset=1)
    assert fs.fs_last_device_error()[0] == fs.FS_ERR_DEVICE_TIMEOUT
    compare(p, dev, offset=1, scores=True)
    assert fs.fs_last_device_error() == (fs.FS_OK, 0)


def test_timeout_read_on_another_stream():
    """The word is one per device: a timeout raised by a kernel on one stream
    is reported by a read ordered on another stream once that kernel is done,
    and the read waits for its own stream only."""
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        fs.fs_wait_timeout_selftest(1_000_000)
    side.synchronize()
    st, code = fs.fs_last_device_error(stream=torch.cuda.current_stream())
    assert st == fs.FS_ERR_DEVICE_TIMEOUT and code & 1
    assert fs.fs_last_device_error(stream=side) == (fs.FS_OK, 0)


def test_selftest_rejects_limits_out_of_range():
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(fs.FsError):
            fs.fs_wait_timeout_selftest(bad)
