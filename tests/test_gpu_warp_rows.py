"""GPU parity of the one-warp-per-row path (many rows of at most 65536 elements).

The path is chosen from 4 to 32 rows per SM on (more for longer rows), so every
batch here has at least that many rows; each test first checks through ds_topk_plan that the call really runs
on that path. Rows are mixed so that the threshold a warp carries from one row
to the next is often wrong (the retry and the exact fallback then run too).
"""
import pytest
import torch

import workloads
from tests.test_gpu_parity import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    torch.cuda.init()
    yield


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _dstk():
    import sampler_topk_selection_ds_b300 as dstk
    return dstk


def _wr_batch(length):
    # the path needs min(32, max(4, len / 1024)) rows per SM; +5 leaves a ragged last CTA
    return min(32, max(4, length // 1024)) * _sms() + 5


def _assert_path(x, k, length=None):
    import sampler_topk_selection_ds_b300 as dstk
    length = x.shape[1] if length is None else length
    dt = dstk.BF16 if x.dtype == torch.bfloat16 else dstk.FP32
    es = x.element_size()
    stride = x.stride(0)
    if stride * es % 16:  # run_gpu pads such rows to a 16-byte stride
        stride = -(-x.shape[1] * es // 16) * 16 // es
    rc, plan = dstk.ds_topk_plan(dt, x.shape[0], length, stride, k, _sms())
    assert rc == 0 and plan.path == dstk.PATH_WARP_ROWS, plan.as_dict()


WR_SHAPES = [
    # (length, k list)
    (1, [1]),
    (7, [1, 7]),
    (100, [1, 37, 100]),
    (1000, [1, 64, 999]),
    (4096, [1, 512, 1024]),
    (4097, [64, 512]),
    (32768, [1, 512, 1024]),
    (65536, [64, 1024]),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("length,ks", WR_SHAPES)
def test_warp_rows_normal(dtype, length, ks):
    x = workloads.random_rows(_wr_batch(length), length, dtype, 500 + length, style="normal")
    for k in ks:
        if dtype == torch.float32 and k > 512 and length > 2304:
            continue  # fp32 with k > 512 on long rows takes the CTA path
        _assert_path(x, k)
        assert_parity(x, k, sorted_index=(k % 2 == 1), return_value=(k % 3 != 2))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("length", [1000, 32768])
def test_warp_rows_mixed_rows(dtype, length):
    """Consecutive rows of one warp differ in scale, offset and structure, so the
    carried threshold fails in both directions; ties, all-equal rows, ramps,
    signed zeros and subnormals force the sample retry and the exact fallback."""
    b = _wr_batch(length)
    styles = ["normal", "ties", "allequal", "ramp", "signed_zero", "denormal"]
    per = b // len(styles) + 1
    parts = [workloads.random_rows(per, length, dtype, 900 + i, style=st)
             for i, st in enumerate(styles)]
    # row r takes style r mod 6, then every row gets its own scale and offset
    x = torch.stack([parts[r % len(styles)][r // len(styles)] for r in range(b)])
    f = x.float()
    shift = (torch.arange(b) % 5).float()[:, None] * 7.0 - 14.0
    scale = 1.0 + (torch.arange(b) % 3).float()[:, None]
    f = torch.where(torch.isfinite(f), f * scale + shift, f)
    x = f.to(dtype).contiguous()
    for k in (1, 64, 512):
        _assert_path(x, k)
        assert_parity(x, k, sorted_index=True, return_value=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_warp_rows_causal_tail_and_nan(dtype):
    """c4-shaped rows (last quarter -inf) with NaN rows spread over the batch."""
    n = 32768
    b = _wr_batch(n)
    x = workloads.random_rows(b, n, dtype, 4242, style="normal")
    x[:, 3 * n // 4:] = float("-inf")
    for r in range(3, b, 97):
        x[r, (r * 131) % n] = float("nan")
    x[b - 1, n - 1] = -float("nan")
    _assert_path(x, 512)
    gv, gi, gf = run_gpu(x, 512, False, True)
    assert gf & 1
    assert_parity(x, 512, False, True, gpu_out=(gv, gi, gf))
    clean = workloads.random_rows(b, n, dtype, 4243, style="normal")
    clean[:, 3 * n // 4:] = float("-inf")
    _, _, gf2 = run_gpu(clean, 512, False, False)
    assert gf2 == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_warp_rows_k_beyond_finite(dtype):
    """k larger than the finite count of a row: -inf elements are selected by index."""
    n = 2048
    b = _wr_batch(n)
    x = workloads.random_rows(b, n, dtype, 77, style="normal")
    x[:, 300:] = float("-inf")
    _assert_path(x, 512)
    assert_parity(x, 512, sorted_index=True, return_value=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_warp_rows_ragged_stride(dtype):
    """len not a multiple of the 16-byte vector, NaN padding that must not be read."""
    es = 2 if dtype == torch.bfloat16 else 4
    for length in (1001, 30001):
        stride = -(-(length + 5) * es // 16) * 16 // es
        x = workloads.random_rows(_wr_batch(length), length, dtype, 31, style="normal", row_stride=stride)
        _assert_path(x, 100, length=length)
        gv, gi, gf = run_gpu(x, 100, True, True, length=length)
        assert gf == 0
        assert_parity(x, 100, True, True, length=length, gpu_out=(gv, gi, gf))


def test_warp_rows_candidates_concentrated():
    """All of a row's large values in one short stretch (recent positions of an
    indexer row), in rows following ordinary rows."""
    n = 32768
    b = _wr_batch(n)
    x = workloads.random_rows(b, n, torch.bfloat16, 5150, style="normal")
    hot = torch.arange(b) % 2 == 1
    x[hot, n - 700:] = (x[hot, n - 700:].float() + 8.0).to(torch.bfloat16)
    _assert_path(x, 512)
    assert_parity(x, 512, sorted_index=False, return_value=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_warp_rows_rows_off_16_byte_boundaries(dtype):
    """Many short rows starting at every element offset within a 16-byte block
    (odd strides, NaN everywhere around the rows, so also inside the first and
    last blocks the kernel reads): the one-warp-per-row path masks every element
    outside a row, so clean rows never raise the NaN flag and match the oracle."""
    from tests.test_gpu_unaligned import place, run_view
    vec = 16 // (2 if dtype == torch.bfloat16 else 4)
    for length, k, style in ((1001, 37, "ties"), (4099, 512, "normal"), (30001, 1000, "normal"),
                             (33, 33, "allequal")):
        b = _wr_batch(length)
        x = workloads.random_rows(b, length, dtype, 6100 + length, style=style)
        for shift, extra in ((1, 1), (vec - 1, 3), (vec // 2, 0)):
            stride = length + extra
            dstk = _dstk()
            dt = dstk.BF16 if dtype == torch.bfloat16 else dstk.FP32
            rc, plan = dstk.ds_topk_plan(dt, b, length, stride, k, _sms())
            assert rc == 0 and plan.path == dstk.PATH_WARP_ROWS
            view = place(x, shift, stride)
            gv, gi, gf = run_view(view, k, sorted_index=bool(shift % 2), return_value=True)
            assert gf == 0
            assert_parity(x, k, bool(shift % 2), True, gpu_out=(gv, gi, gf))


def test_warp_rows_off_boundary_nan_and_causal_tail():
    """Rows off the 16-byte boundary with a -inf tail, and a NaN inside some rows:
    the flag is raised, the clean rows stay exact."""
    from tests.test_gpu_unaligned import place, run_view
    n = 8191
    b = _wr_batch(n)
    x = workloads.random_rows(b, n, torch.bfloat16, 6200, style="normal")
    x[:, 3 * n // 4:] = float("-inf")
    x[5, 0] = float("nan")
    x[9, n - 1] = float("nan")
    view = place(x, 3, n + 1)
    gv, gi, gf = run_view(view, 512, sorted_index=False, return_value=True)
    assert gf & 1
    assert_parity(x, 512, False, True, gpu_out=(gv, gi, gf))


@pytest.mark.parametrize("dtype,length,ks", [
    (torch.bfloat16, 2048, [300, 600, 1024]),    # read whole: the exact k-th element's key
    (torch.bfloat16, 4100, [256, 512, 1000]),    # read whole, ragged
    (torch.bfloat16, 8192, [512, 1024]),         # sampled elements
    (torch.float32, 2304, [300, 512]),           # sampled elements, top 16 key bits
])
def test_warp_rows_dense_k(dtype, length, ks):
    """k over a quarter of the row's 16-byte vectors: thresholds from element
    keys. Ordinary rows, rows of few distinct values (ties at the k-th key
    beyond the candidate room: the exact fallback), and rows whose scale
    changes from one row to the next (the carried threshold fails)."""
    b = _wr_batch(length)
    x = workloads.random_rows(b, length, dtype, 7300 + length, style="normal")
    ties = workloads.random_rows(b, length, dtype, 7301 + length, style="ties")
    x[1::7] = ties[1::7]
    f = x.float()
    scale = 1.0 + (torch.arange(b) % 4).float()[:, None] * 3.0
    x = torch.where(torch.isfinite(f), f * scale, f).to(dtype).contiguous()
    for k in ks:
        _assert_path(x, k)
        assert_parity(x, k, sorted_index=(k % 2 == 0), return_value=True)
