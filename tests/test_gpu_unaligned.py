"""GPU parity of rows that do not start on a 16-byte boundary against the CPU
oracle, bit-exact (every path reads such rows as the 16-byte blocks that
overlap them and masks the elements outside the row).

Rows are placed in a NaN-filled device buffer at an element offset (`shift`)
and with a row stride that need not be a multiple of 16 bytes, so row starts
fall at every offset within a 16-byte vector. The NaN filling surrounds every
row: a clean row must never raise the NaN flag, which checks that no lane
outside the row's [0, len) is ever taken into account.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import bits_of
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    torch.cuda.init()
    yield


def _dstk():
    import sampler_topk_selection_ds_b300 as dstk
    return dstk


def place(x_cpu, shift, stride):
    """A CUDA view of x_cpu [batch, len] whose rows start `shift` elements past a
    16-byte boundary and are `stride` elements apart; NaN everywhere else."""
    batch, length = x_cpu.shape
    assert stride >= length
    buf = torch.full((shift + batch * stride + 16,), float("nan"), dtype=x_cpu.dtype, device="cuda")
    assert buf.data_ptr() % 16 == 0
    view = buf[shift:shift + batch * stride].view(batch, stride)[:, :length]
    view.copy_(x_cpu.cuda())
    return view


def run_view(view, k, sorted_index=False, return_value=True, index_dtype=torch.int32):
    dstk = _dstk()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    vals, idx = dstk.topk(view, k, sorted_index=sorted_index, return_value=return_value,
                          length=view.shape[1], nan_flag=flag, index_dtype=index_dtype)
    torch.cuda.synchronize()
    return (vals.cpu() if vals is not None else None), idx.cpu(), int(flag.item())


def check(x_cpu, k, shift, stride, sorted_index=False, return_value=True):
    view = place(x_cpu, shift, stride)
    assert view.data_ptr() % 16 != 0 or (stride * x_cpu.element_size()) % 16 != 0
    out = run_view(view, k, sorted_index, return_value)
    assert_parity(x_cpu, k, sorted_index, return_value, gpu_out=out)
    return out


def test_plan_reports_the_path():
    dstk = _dstk()
    rc, p = dstk.ds_topk_plan(dstk.BF16, 64, 1001, 1001, 64, 148)
    assert rc == 0 and p.path == dstk.PATH_ROW
    rc, p = dstk.ds_topk_plan(dstk.FP32, 64, 129281, 129281, 512, 148)
    assert rc == 0 and p.path == dstk.PATH_CLUSTER


UA_SWEEP = [
    # (length, batch, k list)
    (1, 3, [1]),
    (7, 5, [1, 3, 7]),
    (9, 5, [1, 9]),
    (33, 4, [1, 5, 33]),
    (1001, 6, [1, 64, 1001]),
    (4096, 3, [1, 512, 4096]),
    (4099, 3, [1, 1024, 4096]),
    (65541, 3, [1, 512, 4096]),
    (129281, 2, [64, 512, 4096]),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("length,batch,ks", UA_SWEEP)
def test_unaligned_sweep(dtype, length, batch, ks):
    x = workloads.random_rows(batch, length, dtype, 40 + length % 97, style="normal")
    vec = 16 // x.element_size()
    for i, k in enumerate(ks):
        shift = (1, vec - 1, vec // 2, 0)[i % 4]
        stride = length + (1, 0, 3, 5)[i % 4]  # odd strides put every row at a new offset
        check(x, k, shift, stride, sorted_index=bool(i % 2))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("style", ["ties", "allequal", "signed_zero", "denormal", "ramp"])
def test_unaligned_adversarial_styles(dtype, style):
    for length, ks in ((37, (1, 10, 37)), (5003, (1, 100, 4096))):
        x = workloads.random_rows(5, length, dtype, 41, style=style)
        for k in ks:
            check(x, k, 1, length + 1, sorted_index=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_many_rows(dtype):
    """More rows than resident CTAs: each CTA walks rows with a stride."""
    x = workloads.random_rows(2000, 300, dtype, 42, style="ties")
    check(x, 37, 3, 301)
    check(x, 300, 0, 303)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_guess_takes_a_bin_whole(dtype):
    """Rows with exactly k elements at 5.0, ten at 4.5 and the rest below 3: from
    the second row on, a CTA guesses the threshold from the previous row, the
    candidates are the k fives, and the radix over them takes a whole 8-bit bin
    whose lower end lies below the guess (the 4.5s share that bin and must not be
    selected)."""
    k = 96
    x = workloads.random_rows(600, 6000, dtype, 48, style="normal").clamp(max=2.9)
    for b in range(x.shape[0]):
        cols = torch.randperm(6000, generator=torch.Generator().manual_seed(b))
        x[b, cols[:k]] = 5.0
        x[b, cols[k:k + 10]] = 4.5
    check(x, k, 1, 6001, sorted_index=True)
    check(x, k + 5, 1, 6001)  # five of the 4.5s by lowest index


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_nan_flag(dtype):
    x = workloads.random_rows(6, 5001, dtype, 43, style="normal")
    x[0, 0] = float("nan")
    x[1, 5000] = float("nan")
    x[2, 2500] = -float("nan")
    x[3, 1000:] = float("-inf")
    x[3, 4000] = float("nan")
    view = place(x, 1, 5001)
    gv, gi, gf = run_view(view, 64, True)
    assert gf & 1
    assert_parity(x, 64, True, True, gpu_out=(gv, gi, gf))  # rows 0-3 skipped, 4-5 exact
    clean = workloads.random_rows(3, 5001, dtype, 44, style="normal")
    assert run_view(place(clean, 1, 5003), 64)[2] == 0  # NaN padding on both sides of every row


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_int64_and_value_order(dtype):
    x = workloads.random_rows(7, 3001, dtype, 45, style="ties")
    k = 200
    view = place(x, 1, 3003)
    ov, oi, _, _ = oracle.topk(x, k, return_value=True, order="value")
    for rv in (True, False):
        gv, gi, gf = run_view(view, k, "value", rv, index_dtype=torch.int64)
        assert gf == 0 and gi.dtype == torch.int64
        assert torch.equal(gi, oi.to(torch.int64))
        if rv:
            assert np.array_equal(bits_of(gv), bits_of(ov))
    _, oi_idx, _, _ = oracle.topk(x, k)
    _, gi, _ = run_view(view, k, True, False, index_dtype=torch.int64)
    assert torch.equal(gi, oi_idx.to(torch.int64))


def test_unaligned_sampler():
    from tests.test_gpu_sampler import check_sample
    x = workloads.random_rows(9, 1003, torch.float32, 46, style="normal")
    check_sample(x, 64, 0.8, 0.9, 12, xd=place(x, 1, 1003))
    xb = workloads.random_rows(9, 1003, torch.bfloat16, 47, style="normal")
    check_sample(xb, 256, 1.0, 0.95, 13, xd=place(xb, 3, 1005))


def test_unaligned_c2_shape_full():
    """The sampler workload's shape (64 x 129280 fp32, k = 512) one element off
    the 16-byte boundary: every row checked against the oracle."""
    w = workloads.WORKLOADS["c2"]
    x = workloads.generate(w)
    check(x, w.k, 1, w.length, w.sorted_index, w.return_value)


def test_unaligned_c4_shape_full():
    """The decode workload's shape (16384 x 32768 bf16, k = 512) one element off
    the 16-byte boundary, as the benchmark's shifted mode times it: every row
    against the oracle."""
    from tests.test_gpu_parity import assert_rows_equal_oracle
    w = workloads.WORKLOADS["c4"]
    xd = workloads.generate(w, device="cuda")
    buf = torch.empty(w.batch * w.length + 8, dtype=xd.dtype, device="cuda")
    view = buf[1:1 + w.batch * w.length].view(w.batch, w.length)
    view.copy_(xd)
    del xd
    gv, gi, gf = run_view(view, w.k, w.sorted_index, w.return_value)
    assert gv is None and gf == 0
    x = view.cpu()
    del buf, view
    assert_rows_equal_oracle(x, w.k, gi)
