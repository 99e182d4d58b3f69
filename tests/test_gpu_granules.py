"""GPU parity where the launch plan groups several 16-byte vectors into one
granule (long rows in many-row batches: a CTA per row, or a 2-CTA cluster).

Rows of a few repeated values (ties, signed zeros, all equal) send the
selection to its fallback over the listed granules, where the ties at the k-th
key are taken in index order across granules and across the vectors inside a
granule; for sorted_index 1 every output must also be in ascending index order.
"""
import pytest
import torch

import workloads
from tests.test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    torch.cuda.init()
    yield


@pytest.mark.parametrize("dtype,batch,length,gv", [
    (torch.bfloat16, 300, 70001, 2),   # CTA per row
    (torch.float32, 148, 70001, 2),    # 2-CTA clusters
    (torch.float32, 300, 70001, 3),    # CTA per row, ragged last granule
])
def test_multi_vector_granules(dtype, batch, length, gv):
    import sampler_topk_selection_ds_b300 as dstk
    dt = dstk.BF16 if dtype == torch.bfloat16 else dstk.FP32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    parts = [workloads.random_rows(batch, length, dtype, 8100 + i, style=st)
             for i, st in enumerate(("signed_zero", "ties", "normal", "allequal"))]
    x = torch.stack([parts[r % 4][r] for r in range(batch)])
    for k in (1, 7, 64, 1000):
        rc, plan = dstk.ds_topk_plan(dt, batch, length, length, k, sms)
        assert rc == 0 and plan.vectors_per_granule == gv, plan.as_dict()
        for sorted_index in (True, False):
            assert_parity(x, k, sorted_index=sorted_index, return_value=(k != 7))
