"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit-exact.

Indices and values must equal the oracle's exactly (selection does no
arithmetic). With sorted_index=0 the order is unspecified by contract, so both
sides are compared after sorting by index; with sorted_index=1 the GPU order
itself must be ascending. Rows holding a NaN are only checked for the flag and
for in-range outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import bits_of, check_invariants

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


def _aligned(x, length):
    """Rows whose byte length is not a multiple of 16 are copied into a padded
    buffer (NaN padding, which must never be read), so that these tests run the
    paths for rows on 16-byte boundaries; rows off those boundaries are covered
    by test_gpu_unaligned.py and test_gpu_warp_rows.py."""
    es = x.element_size()
    if x.stride(0) * es % 16 == 0 or x.shape[0] == 1:
        return x, length
    stride = -(-x.shape[1] * es // 16) * 16 // es
    xp = torch.full((x.shape[0], stride), float("nan"), dtype=x.dtype, device=x.device)
    xp[:, :x.shape[1]] = x
    return xp, x.shape[1] if length is None else length


def run_gpu(x, k, sorted_index, return_value, length=None, stream=None):
    dstk = _dstk()
    x, length = _aligned(x, length)
    xd = x if x.is_cuda else x.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device=xd.device)
    vals, idx = dstk.topk(xd, k, sorted_index=sorted_index, return_value=return_value,
                          length=length, nan_flag=flag, stream=stream)
    torch.cuda.synchronize()
    return (vals.cpu() if vals is not None else None), idx.cpu(), int(flag.item())


def assert_parity(x_cpu, k, sorted_index=False, return_value=True, length=None, rows=None,
                  gpu_out=None):
    """Compare GPU output with the oracle on rows `rows` (all rows by default)."""
    length = x_cpu.shape[1] if length is None else length
    if gpu_out is None:
        gv, gi, gf = run_gpu(x_cpu, k, sorted_index, return_value, length)
    else:
        gv, gi, gf = gpu_out
    sel = list(range(x_cpu.shape[0])) if rows is None else list(rows)
    ov, oi, of, row_nan = oracle.topk(x_cpu[sel].contiguous(), k, length=length, return_value=True)
    if rows is None:
        assert gf == of, f"nan flag gpu={gf} oracle={of}"
    for j, b in enumerate(sel):
        g_idx = gi[b].numpy().astype(np.int64)
        assert g_idx.min() >= 0 and g_idx.max() < length
        if row_nan[j]:
            continue
        if sorted_index:
            assert np.all(np.diff(g_idx) > 0), f"row {b}: sorted_index output not ascending"
            order = np.arange(k)
        else:
            order = np.argsort(g_idx, kind="stable")
        o_idx = oi[j].numpy().astype(np.int64)
        if not np.array_equal(g_idx[order], o_idx):
            bad = np.nonzero(g_idx[order] != o_idx)[0]
            raise AssertionError(f"row {b}: {bad.size} index mismatches, first at {bad[0]}: "
                                 f"gpu {g_idx[order][bad[0]]} oracle {o_idx[bad[0]]}")
        if return_value:
            assert np.array_equal(bits_of(gv[b])[order], bits_of(ov[j])), f"row {b}: values differ"


# ---- the five workloads at full size ---------------------------------------------------

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
def test_workload_full_parity(name):
    w = workloads.WORKLOADS[name]
    x = workloads.generate(w)
    assert_parity(x, w.k, w.sorted_index, w.return_value)


def assert_rows_equal_oracle(x_cpu, k, gi, gv=None, order="index"):
    """Every row of a GPU result against the oracle on all host threads, compared
    as whole tensors: indices (canonically sorted by index unless order="value",
    where the position is part of the result) and, if given, the value bits at
    the same positions. Rows holding a NaN are not expected here."""
    ov, oi, of, row_nan = oracle.topk(x_cpu, k, return_value=gv is not None, order=order)
    assert of == 0 and not row_nan.any()
    gi64 = gi.to(torch.int64)
    if order == "value":
        perm = torch.arange(k).expand_as(gi64)
    else:
        perm = torch.argsort(gi64, dim=1, stable=True)
    g_sorted = torch.gather(gi64, 1, perm)
    bad = (g_sorted != oi.to(torch.int64)).any(dim=1).nonzero().flatten()
    assert bad.numel() == 0, f"{bad.numel()} rows differ from the oracle, first row {int(bad[0])}"
    if gv is not None:
        gb = torch.from_numpy(bits_of(gv).astype(np.int64))
        ob = torch.from_numpy(bits_of(ov).astype(np.int64))
        assert torch.equal(torch.gather(gb, 1, perm), ob), "value bits differ from the oracle"


def test_workload_c4_full_parity():
    """c4 (16384 x 32768 bf16, indices only): the whole batch on the GPU in the
    benchmark's launch configuration, every row against the oracle. These rows
    drive the one-warp-per-row path's threshold guesses and retries, where a rare
    wrong row would hide."""
    w = workloads.WORKLOADS["c4"]
    xd = workloads.generate(w, device="cuda")
    gv, gi, gf = run_gpu(xd, w.k, w.sorted_index, w.return_value)
    assert gv is None and gf == 0
    x = xd.cpu()
    del xd
    assert_rows_equal_oracle(x, w.k, gi)


def test_workload_c4_full_value_order():
    """c4's batch with value-ordered output and values returned: every row's
    positions, indices and value bits equal the oracle's value order."""
    w = workloads.WORKLOADS["c4"]
    xd = workloads.generate(w, device="cuda")
    gv, gi, gf = run_gpu(xd, w.k, "value", True)
    assert gf == 0
    x = xd.cpu()
    del xd
    assert_rows_equal_oracle(x, w.k, gi, gv, order="value")


# ---- sweeps ------------------------------------------------------------------------------

SWEEP = [
    # (length, batch, k list)
    (1, 3, [1]),
    (7, 3, [1, 2, 7]),
    (31, 5, [1, 2, 31]),
    (4096, 3, [1, 2, 64, 512, 1024, 4095, 4096]),
    (4097, 3, [1, 64, 4096]),
    (65541, 3, [1, 512, 4096]),
    (129280, 3, [64, 512, 4096]),
    (204800, 2, [1024, 4096]),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("length,batch,ks", SWEEP)
def test_sweep_normal(dtype, length, batch, ks):
    x = workloads.random_rows(batch, length, dtype, 1000 + length, style="normal")
    for k in ks:
        assert_parity(x, k, sorted_index=(k % 2 == 0), return_value=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("style", ["ties", "allequal", "signed_zero", "denormal", "ramp"])
@pytest.mark.parametrize("length", [33, 4096, 70001])
def test_sweep_adversarial_styles(dtype, style, length):
    x = workloads.random_rows(3, length, dtype, 77, style=style)
    for k in sorted({1, min(64, length), min(4096, length), min(length, 4096)}):
        assert_parity(x, k, sorted_index=True, return_value=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_row_stride_padding_and_tail(dtype):
    # len not a multiple of the 16-byte vector, padding filled with NaN (never read)
    for length, stride in [(5, 8), (1001, 1024), (65537, 65600)]:
        es = 2 if dtype == torch.bfloat16 else 4
        stride = -(-stride * es // 16) * 16 // es
        x = workloads.random_rows(4, length, dtype, 5, style="normal", row_stride=stride)
        k = min(100, length)
        gv, gi, gf = run_gpu(x, k, True, True, length=length)
        assert gf == 0
        assert_parity(x, k, True, True, length=length, gpu_out=(gv, gi, gf))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_batch_many_short_rows(dtype):
    x = workloads.random_rows(3000, 1000, dtype, 11, style="ties")
    assert_parity(x, 37, sorted_index=False, return_value=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_long_single_row_coarse_granules(dtype):
    """A row long enough that each cluster CTA summarises several vectors per granule."""
    n = (1 << 23) + 3 if dtype == torch.float32 else (1 << 24) + 5
    x = workloads.random_rows(1, n, dtype, 3, style="normal")
    assert_parity(x, 4096, sorted_index=True, return_value=True)
    assert_parity(x, 1, sorted_index=True, return_value=False)


def test_values_skipped_and_nonnull_untouched():
    w = workloads.WORKLOADS["c1"]
    x = workloads.generate(w).cuda()
    dstk = _dstk()
    sentinel = torch.full((w.batch, w.k), -12345.0, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty((w.batch, w.k), dtype=torch.int32, device="cuda")
    rc = dstk.ds_topk(x.data_ptr(), dstk.FP32, w.batch, w.length, w.length, w.k, 0, 0,
                      sentinel.data_ptr(), idx.data_ptr(), flag.data_ptr(), 0)
    torch.cuda.synchronize()
    assert rc == 0
    assert (sentinel == -12345.0).all(), "out_values written although return_value == 0"
    _, oi, _, _ = oracle.topk(x.cpu(), w.k)
    assert torch.equal(torch.sort(idx.cpu(), dim=1).values, oi)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_nan_flag_and_clean_rows_exact(dtype):
    for length in (4096, 300000):
        x = workloads.random_rows(6, length, dtype, 21, style="normal")
        x[0, 0] = float("nan")
        x[1, length // 2] = float("nan")
        x[2, length - 1] = float("nan")
        x[3, length // 3:] = float("-inf")
        x[3, length - 2] = float("nan")       # NaN inside a -inf tail
        x[4, 3] = -float("nan")               # negative NaN never beats any threshold
        gv, gi, gf = run_gpu(x, 64, True, True)
        assert gf & 1
        assert_parity(x, 64, True, True, gpu_out=(gv, gi, gf))  # rows 0-4 skipped, row 5 exact
        clean = workloads.random_rows(2, length, dtype, 22, style="normal")
        _, _, gf2 = run_gpu(clean, 64, True, True)
        assert gf2 == 0


def test_flag_is_sticky_and_not_cleared():
    dstk = _dstk()
    x = workloads.random_rows(2, 1000, torch.float32, 1).cuda()
    flag = torch.full((1,), 4, dtype=torch.int32, device="cuda")  # caller's own bit
    dstk.topk(x, 10, nan_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 4


def test_batch_zero_and_stream():
    dstk = _dstk()
    rc = dstk.ds_topk(0, dstk.BF16, 0, 100, 128, 5, 0, 0, None, 0, 0, 0)
    assert rc == dstk.OK
    s = torch.cuda.Stream()
    x = workloads.random_rows(4, 5000, torch.bfloat16, 9)
    with torch.cuda.stream(s):
        gv, gi, gf = run_gpu(x, 300, False, True, stream=s)
    assert_parity(x, 300, False, True, gpu_out=(gv, gi, gf))


def test_invariants_on_gpu_output_c3():
    w = workloads.WORKLOADS["c3"]
    x = workloads.generate(w)
    gv, gi, gf = run_gpu(x, w.k, True, True)
    for b in range(w.batch):
        check_invariants(x[b], w.k, gi[b].numpy(), bits_of(gv[b]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_k_beyond_finite_granules(dtype):
    """k above the number of vectors holding a finite value: the granule threshold is
    -inf, every element is a candidate, and the selection must still resolve the
    k-th key directly (one CTA per row, and a cluster per row)."""
    x = workloads.random_rows(64, 4096, dtype, 4096, style="normal")
    x[:, 3072:] = float("-inf")          # 3072 finite values, 384 (bf16) / 768 (fp32) vectors
    for k in (512, 1024):
        assert_parity(x, k, sorted_index=False, return_value=True)
    x = workloads.random_rows(2, 300000, dtype, 4097, style="normal")
    x[:, 2000:] = float("-inf")
    assert_parity(x, 4096, sorted_index=True, return_value=True)


def test_concurrent_streams():
    """Calls on different streams may overlap (the library keeps no global
    scratch): one CTA per row, a cluster per row, one warp per row and the value
    order, all enqueued before any synchronisation."""
    dstk = _dstk()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [
        (workloads.random_rows(8, 4096, torch.float32, 801), 64, True),
        (workloads.random_rows(2, 300000, torch.bfloat16, 802), 1024, True),
        (workloads.random_rows(4 * sms + 1, 1000, torch.bfloat16, 803, style="ties"), 37, True),
        (workloads.random_rows(16, 50000, torch.float32, 804), 512, "value"),
    ]
    streams = [torch.cuda.Stream() for _ in cases]
    devs = [x.cuda() for x, _, _ in cases]
    torch.cuda.synchronize()
    outs = []
    for (x, k, order), xd, s in zip(cases, devs, streams):
        with torch.cuda.stream(s):
            outs.append(dstk.topk(xd, k, sorted_index=order, return_value=True, stream=s))
    torch.cuda.synchronize()
    for (x, k, order), (gv, gi) in zip(cases, outs):
        ov, oi, _, _ = oracle.topk(x, k, order="value" if order == "value" else "index")
        assert torch.equal(gi.cpu(), oi)
        assert np.array_equal(bits_of(gv.cpu()), bits_of(ov))
