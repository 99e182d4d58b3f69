"""The bounded mbarrier wait of the one-warp-per-row kernel gives up cleanly.

A probe (tests/wait_timeout_probe.cu) is compiled with a short poll limit and
waits on an mbarrier phase that nothing completes and no copy feeds: the wait
must return, the kernel must raise DS_TOPK_FLAG_TIMEOUT in the status word, and
the context must stay usable. A phase that does complete must not raise it.
Nothing here hangs or faults a GPU: every wait is bounded by the poll limit.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "sampler_topk_selection_ds_b300", "csrc")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
LIMIT = 64


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    torch.cuda.init()
    out = os.path.join(tempfile.mkdtemp(prefix="ds_topk_wait_"), "libwait_probe.so")
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", f"-DDS_TOPK_WAIT_LIMIT={LIMIT}u", f"-I{os.path.join(ROOT, 'include')}",
           f"-I{CSRC}", "--expt-relaxed-constexpr", "-o", out, os.path.join(HERE, "wait_timeout_probe.cu")]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.wait_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.wait_probe.restype = ctypes.c_int
    lib.wait_probe_limit.restype = ctypes.c_uint
    return lib


def test_wait_runs_out_and_sets_timeout_flag(probe):
    import sampler_topk_selection_ds_b300 as dstk
    assert probe.wait_probe_limit() == LIMIT
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert probe.wait_probe(0, flag.data_ptr(), waited.data_ptr()) == 0
    assert int(waited.item()) == 1, "the kernel did not return from the wait"
    assert int(flag.item()) == dstk.FLAG_TIMEOUT
    # the context is still usable: a TopK call runs and is exact afterwards
    x = torch.randn(4, 4096, device="cuda")
    _, idx = dstk.topk(x, 16, sorted_index=True)
    ref = torch.sort(torch.topk(x, 16, dim=1).indices, dim=1).values
    assert torch.equal(idx.to(torch.int64), ref)


def test_completed_phase_does_not_time_out(probe):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert probe.wait_probe(1, flag.data_ptr(), waited.data_ptr()) == 0
    assert int(waited.item()) == 1 and int(flag.item()) == 0
