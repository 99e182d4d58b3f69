"""GPU parity with int64 output indices (ds_topk_ex, DS_TOPK_INDEX_INT64) on
every launch path: the same selection as the oracle, written as int64."""
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


def check_i64(x, k, order):
    import sampler_topk_selection_ds_b300 as dstk
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    gv, gi = dstk.topk(x.cuda(), k, sorted_index=order, return_value=True, nan_flag=flag,
                       index_dtype=torch.int64)
    torch.cuda.synchronize()
    assert gi.dtype == torch.int64
    ov, oi, of, row_nan = oracle.topk(x, k, order="value" if order == "value" else "index")
    assert int(flag.item()) == of and not bool(row_nan.any())
    assert torch.equal(gi.cpu(), oi.to(torch.int64))
    assert np.array_equal(bits_of(gv.cpu()), bits_of(ov))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("order", [True, "value"])
def test_int64_indices_every_path(dtype, order):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    check_i64(workloads.random_rows(8, 4096, dtype, 71, style="ties"), 300, order)        # CTA per row
    check_i64(workloads.random_rows(2, 300000, dtype, 72, style="normal"), 4096, order)   # cluster
    check_i64(workloads.random_rows(4 * sms + 3, 1000, dtype, 73, style="normal"), 64, order)  # warp rows
    # many rows: for bf16 and value order also the one-warp-per-row sort
    check_i64(workloads.random_rows(8 * sms + 3, 1000, dtype, 74, style="ties"), 300, order)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_int64_indices_value_order_without_values(dtype):
    """Value order with int64 indices and no values: the sort gathers the keys from
    x (one warp per row for the bf16 batch of 8 rows per SM, one CTA per row else)."""
    import sampler_topk_selection_ds_b300 as dstk
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for batch, k in ((8 * sms + 3, 300), (8, 1000)):
        x = workloads.random_rows(batch, 1000 if batch > 8 else 4096, dtype, 75 + k, style="signed_zero")
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        _, gi = dstk.topk(x.cuda(), k, sorted_index="value", return_value=False, nan_flag=flag,
                          index_dtype=torch.int64)
        torch.cuda.synchronize()
        _, oi, of, row_nan = oracle.topk(x, k, order="value")
        assert int(flag.item()) == of and not bool(row_nan.any())
        assert gi.dtype == torch.int64 and torch.equal(gi.cpu(), oi.to(torch.int64))

