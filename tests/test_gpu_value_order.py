"""GPU parity of the value-ordered output (sorted_index = DS_TOPK_SORT_VALUE).

Each output row must equal the oracle's value order exactly: indices and value
bits in the same positions (value descending, equal values by ascending index),
on all three launch paths (one CTA per row, a cluster per row, one warp per row).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import bits_of

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


def _path(x, k):
    dstk = _dstk()
    dt = dstk.BF16 if x.dtype == torch.bfloat16 else dstk.FP32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, plan = dstk.ds_topk_plan(dt, x.shape[0], x.shape[1], x.stride(0), k, sms)
    assert rc == 0
    return plan.path


def check_value_order(x, k, return_value=True):
    dstk = _dstk()
    xd = x.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    gv, gi = dstk.topk(xd, k, sorted_index="value", return_value=return_value, nan_flag=flag)
    torch.cuda.synchronize()
    ov, oi, of, row_nan = oracle.topk(x, k, order="value")
    assert int(flag.item()) == of
    gi = gi.cpu()
    assert int(gi.min()) >= 0 and int(gi.max()) < x.shape[1]
    keep = ~row_nan
    assert torch.equal(gi[keep], oi[keep]), "value order differs from the oracle"
    if return_value:
        assert np.array_equal(bits_of(gv.cpu()[keep]), bits_of(ov[keep]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("style", ["normal", "ties", "signed_zero", "allequal"])
def test_value_order_cta_path(dtype, style):
    x = workloads.random_rows(8, 4096, dtype, 612, style=style)
    assert _path(x, 64) == _dstk().PATH_ROW
    for k in (1, 64, 1000, 4096):
        check_value_order(x, k, return_value=(k != 1000))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_value_order_cluster_path(dtype):
    x = workloads.random_rows(2, 300000, dtype, 613, style="normal")
    assert _path(x, 512) == _dstk().PATH_CLUSTER
    for k in (512, 4096):
        check_value_order(x, k)
    w = workloads.WORKLOADS["c2"] if dtype == torch.float32 else workloads.WORKLOADS["c3"]
    check_value_order(workloads.generate(w), w.k)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_value_order_warp_rows_path(dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x = workloads.random_rows(4 * sms + 3, 1000, dtype, 614, style="ties")
    assert _path(x, 37) == _dstk().PATH_WARP_ROWS
    for k in (1, 37, 512):
        check_value_order(x, k, return_value=(k != 512))
    n = 32768
    x = workloads.random_rows(32 * sms + 1, n, dtype, 615, style="normal")
    x[:, 3 * n // 4:] = float("-inf")
    assert _path(x, 512) == _dstk().PATH_WARP_ROWS
    check_value_order(x, 512, return_value=False)


def test_value_order_nan_rows_in_range():
    x = workloads.random_rows(6, 5000, torch.bfloat16, 616, style="normal")
    x[2, 17] = float("nan")
    check_value_order(x, 300)  # the NaN row is only checked for the flag and in-range indices


ALL_WIDTHS = (1, 2, 31, 32, 33, 64, 65, 100, 128, 129, 256, 257, 300, 511, 512, 513, 1000, 1024, 1025)


@pytest.mark.parametrize("dtype,n,ks", [(torch.bfloat16, 3000, ALL_WIDTHS),
                                        (torch.bfloat16, 65536, (1, 33, 512, 1024)),
                                        (torch.bfloat16, 70001, (1, 33, 512, 1024)),
                                        (torch.float32, 3000, (1, 33, 512, 1024, 1025))])
def test_value_order_register_sort_widths(dtype, n, ks):
    """Many bf16 rows of at most 65536 elements with k <= 1024 sort one row per
    warp in registers, n2 / 32 words per lane for n2 = k rounded up to a power of
    two (at least 32): every width from 1 to 32 words, and the k just above 1024
    that goes back to the CTA sort. 32-bit sort words hold a 16-bit index, so the
    last index of a 65536-element row complements to 0. Longer bf16 rows and fp32
    rows keep the CTA sort with 64-bit words. Ties and signed zeros throughout."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    b = 8 * sms + 3 if dtype == torch.bfloat16 and n <= 65536 else 40  # the warp sort needs 8 rows per SM
    x = workloads.random_rows(b, n, dtype, 617 + n, style="signed_zero")
    x[1::2] = workloads.random_rows(b, n, dtype, 618 + n, style="ties")[1::2]
    x[5, n - 1] = 3e38  # a ties row's largest element at its last index
    for k in ks:
        check_value_order(x, k, return_value=(k % 2 == 0))
