"""The C-ABI boundary on the CPU: the library loads, exports every symbol the
header declares, rejects bad arguments with the documented code before touching
the GPU, and plans launches as documented. No call here reaches a kernel."""
import ctypes
import os
import re

import pytest

import sampler_topk_selection_ds_b300 as dstk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn), encoding="utf-8").read()
            names |= set(re.findall(r"DS_TOPK_API\s+[\w\s\*]*?\b(ds_topk\w*)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    names = _declared_symbols()
    assert {"ds_topk", "ds_topk_plan", "ds_topk_status_string", "ds_topk_version"} <= names
    lib = ctypes.CDLL(dstk.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings():
    assert dstk.version() >= 100
    assert dstk.status_string(dstk.OK) == "ok"
    assert "invalid" in dstk.status_string(dstk.EINVAL)
    assert "align" in dstk.status_string(dstk.EALIGN)
    assert dstk.status_string(99) == "unknown status"


# Pointers below are never dereferenced: every call fails validation first.
P = 1 << 20  # a 16-byte-aligned fake address


@pytest.mark.parametrize("args,code", [
    # (x, dtype, batch, len, row_stride, k, sorted, retval, out_values, out_indices, flag)
    ((P, 2, 1, 16, 16, 1, 0, 1, P, P, P), dstk.EINVAL),          # bad dtype
    ((P, 0, -1, 16, 16, 1, 0, 1, P, P, P), dstk.EINVAL),         # negative batch
    ((P, 0, 1, 0, 16, 1, 0, 1, P, P, P), dstk.EINVAL),           # len 0
    ((P, 0, 1, 2**31, 2**31, 1, 0, 1, P, P, P), dstk.EINVAL),    # len > INT32_MAX
    ((P, 0, 1, 16, 8, 1, 0, 1, P, P, P), dstk.EINVAL),           # row_stride < len
    ((P, 0, 1, 16, 16, 0, 0, 1, P, P, P), dstk.EINVAL),          # k = 0
    ((P, 0, 1, 8192, 8192, 4097, 0, 1, P, P, P), dstk.EINVAL),   # k > 4096
    ((P, 0, 1, 16, 16, 17, 0, 1, P, P, P), dstk.EINVAL),         # k > len
    ((P, 0, 1, 16, 16, 1, 3, 1, P, P, P), dstk.EINVAL),          # sorted_index not 0/1/2
    ((P, 0, 1, 16, 16, 1, 0, 3, P, P, P), dstk.EINVAL),          # return_value not 0/1
    ((0, 0, 1, 16, 16, 1, 0, 1, P, P, P), dstk.EINVAL),          # x NULL
    ((P, 0, 1, 16, 16, 1, 0, 1, P, 0, P), dstk.EINVAL),          # out_indices NULL
    ((P, 0, 1, 16, 16, 1, 0, 1, P, P, 0), dstk.EINVAL),          # nan_flag NULL
    ((P, 0, 1, 16, 16, 1, 0, 1, 0, P, P), dstk.EINVAL),          # values requested, NULL
    ((P + 1, 0, 1, 16, 16, 1, 0, 1, P, P, P), dstk.EALIGN),      # bf16 x not 2-byte aligned
    ((P + 2, 1, 1, 16, 16, 1, 0, 1, P, P, P), dstk.EALIGN),      # fp32 x not 4-byte aligned
    ((P, 0, 1, 16, 16, 1, 0, 1, P, P + 2, P), dstk.EALIGN),      # out_indices misaligned
    ((P, 0, 1, 16, 16, 1, 0, 1, P, P, P + 1), dstk.EALIGN),      # flag misaligned
    ((P, 1, 1, 16, 16, 1, 0, 1, P + 2, P, P), dstk.EALIGN),      # fp32 values misaligned
    ((P, 0, 2**40, 2**30, 2**30, 1, 0, 1, P, P, P), dstk.EINVAL),  # batch*stride overflows
])
def test_argument_errors(args, code):
    assert dstk.ds_topk(*args, 0) == code


def test_batch_zero_is_ok_without_pointers():
    assert dstk.ds_topk(0, dstk.BF16, 0, 100, 128, 5, 0, 0, None, 0, 0, 0) == dstk.OK


def test_plan_shapes():
    # many short rows: one warp per row, 8 rows per CTA, ~2k candidate slots per warp
    rc, p = dstk.ds_topk_plan(dstk.BF16, 16384, 32768, 32768, 512, 148)
    assert rc == 0 and p.path == dstk.PATH_WARP_ROWS and p.cluster_size == 1
    assert p.grid_ctas == 16384 // 8 and p.threads_per_cta == 256 and p.launches == 1
    assert p.granules_per_cta == 1024 and 3 * (p.smem_bytes + 1024) <= 228 * 1024  # 3 CTAs per SM
    # fewer than 8 rows per SM: one CTA per row
    rc, p = dstk.ds_topk_plan(dstk.BF16, 1000, 32768, 32768, 512, 148)
    assert rc == 0 and p.path == dstk.PATH_ROW and p.grid_ctas == 1000
    assert p.vectors_per_granule == 1
    # warp path limits: 16-bit candidate indices, and its shared memory
    assert dstk.ds_topk_plan(dstk.BF16, 4096, 65537, 65544, 512, 148)[1].path == dstk.PATH_ROW
    assert dstk.ds_topk_plan(dstk.BF16, 4096, 65536, 65536, 2048, 148)[1].path == dstk.PATH_ROW
    assert dstk.ds_topk_plan(dstk.FP32, 4096, 65536, 65536, 1024, 148)[1].path == dstk.PATH_ROW
    rc, p = dstk.ds_topk_plan(dstk.FP32, 4096, 100, 100, 100, 148)
    assert rc == 0 and p.path == dstk.PATH_WARP_ROWS and p.granules_per_cta == 128
    rc, p = dstk.ds_topk_plan(dstk.FP32, 64, 129280, 129280, 512, 148)
    assert rc == 0 and p.path == dstk.PATH_CLUSTER and p.cluster_size in (2, 4, 8, 16)
    assert p.grid_ctas == 64 * p.cluster_size
    rc, p = dstk.ds_topk_plan(dstk.BF16, 8, 1 << 20, 1 << 20, 4096, 148)
    assert rc == 0 and p.cluster_size == 16 and p.granules_per_cta <= 8192
    rc, p = dstk.ds_topk_plan(dstk.FP32, 1, (1 << 23) + 3, (1 << 23) + 4, 4096, 148)
    assert rc == 0 and p.cluster_size == 16 and p.vectors_per_granule > 1
    assert p.granules_per_cta <= 8192
    rc, p = dstk.ds_topk_plan(dstk.FP32, 0, 100, 100, 5, 148)
    assert rc == 0 and p.launches == 0
    # small rows are never split
    rc, p = dstk.ds_topk_plan(dstk.FP32, 4, 4096, 4096, 64, 148)
    assert rc == 0 and p.cluster_size == 1
    # validation is shared with ds_topk
    assert dstk.ds_topk_plan(dstk.FP32, 1, 10, 10, 11, 148)[0] == dstk.EINVAL
    assert dstk.ds_topk_plan(dstk.FP32, 1, 10, 12, 5, 0)[0] == dstk.EINVAL

def test_plan_unaligned_rows():
    """Row strides that are not a multiple of 16 bytes put rows off 16-byte
    boundaries. Every path reads such rows as the 16-byte blocks that overlap
    them, so the path is chosen from the sizes alone, as for aligned rows: many
    short rows take one warp per row, others one CTA or cluster per row, with
    up to one block more per row and no next-row prefetch."""
    for dtype, stride in ((dstk.BF16, 10), (dstk.BF16, 32769), (dstk.FP32, 6), (dstk.FP32, 129281)):
        es = 2 if dtype == dstk.BF16 else 4
        for batch, k in ((2, 5), (16384, 512), (64, 4)):
            length = stride if stride > 10 else stride - 1
            kk = min(k, length)
            rc, p = dstk.ds_topk_plan(dtype, batch, length, stride, kk, 148)
            assert rc == 0
            warp_rows = length <= 65536 and kk <= 1024 and batch >= min(32, max(4, length // 1024)) * 148
            if warp_rows:
                assert p.path == dstk.PATH_WARP_ROWS, (dtype, stride, batch)
                continue
            assert p.path in (dstk.PATH_ROW, dstk.PATH_CLUSTER), (dtype, stride, batch)
            # the CTAs' slices cover every 16-byte block a row off the boundary can overlap
            vec = 16 // es
            blocks = -(-(length + vec - 1) // vec)
            assert p.cluster_size * p.granules_per_cta * p.vectors_per_granule >= blocks
    rc, p = dstk.ds_topk_plan(dstk.BF16, 2, 10, 16, 5, 148)  # 32-byte stride
    assert rc == 0 and p.path == dstk.PATH_ROW
    rc, p = dstk.ds_topk_plan(dstk.FP32, 0, 10, 10, 5, 148)
    assert rc == 0 and p.launches == 0


def test_binding_has_no_cpu_fallback():
    import torch
    with pytest.raises(ValueError):
        dstk.topk(torch.zeros(2, 16), 3)


def test_index_type_checks():
    P = 1 << 20  # fake 16-byte aligned device address, never dereferenced
    base = (P, dstk.FP32, 2, 16, 16, 4, 0, 1)
    # an index type other than int32 / int64 is rejected before anything runs
    for bad in (-1, 2, 7):
        assert dstk.ds_topk_ex(*base, bad, P, P, P, 0) == dstk.EINVAL
    # int64 indices need 8-byte alignment
    assert dstk.ds_topk_ex(*base, dstk.INDEX_INT64, P, P + 4, P, 0) == dstk.EALIGN
    assert dstk.ds_topk_ex(0, dstk.FP32, 0, 16, 16, 4, 0, 0, dstk.INDEX_INT64, 0, 0, 0, 0) == dstk.OK


def test_bench_shift_layout_and_plan():
    """bench.py --shift: the copy sits `shift` elements past an aligned start with
    the same contents; each workload keeps its path at any shift (the decode-
    shaped batch one warp per row, the sampler's long rows a cluster per row)."""
    import torch

    import bench
    import workloads
    x = torch.arange(24, dtype=torch.float32).view(4, 6)
    for shift in (0, 1, 3):
        y = bench.shifted(x, shift)
        assert torch.equal(y, x) and y.stride() == x.stride()
        if shift == 0:
            assert y.data_ptr() == x.data_ptr()  # no copy
        else:
            assert y.data_ptr() % 16 == shift * 4 % 16  # the buffer's start is 16-byte aligned
    c4 = workloads.WORKLOADS["c4"]  # bf16 rows of 65536 bytes
    for shift, path in ((0, dstk.PATH_WARP_ROWS), (1, dstk.PATH_WARP_ROWS), (7, dstk.PATH_WARP_ROWS),
                        (8, dstk.PATH_WARP_ROWS)):
        rc, p = bench.plan_for(dstk, c4, 148, shift)
        assert rc == dstk.OK and p.path == path, (shift, p.path)
        assert bench.kernel_name(c4, p).startswith("topk_warp_rows")
    c2 = workloads.WORKLOADS["c2"]  # fp32: a 4-element shift keeps 16-byte alignment
    assert bench.plan_for(dstk, c2, 148, 4)[1].path == dstk.PATH_CLUSTER
    assert bench.plan_for(dstk, c2, 148, 2)[1].path == dstk.PATH_CLUSTER


def test_bench_kernel_hash_ignores_comments_only():
    """The hash that ties a profile's DRAM traffic to a kernel covers code, not
    comments or layout: a comment edit keeps it, a code edit changes it."""
    import bench
    base = 'int f(int a) { return a + 1; } // one\nconst char* s = "a // b";\n'
    assert bench.code_only(base) == bench.code_only(
        '/* a note */ int f(int a)  {\n  return a + 1;  // two\n}\nconst char* s = "a // b";')
    assert bench.code_only(base) != bench.code_only(base.replace("a + 1", "a + 2"))
    assert bench.code_only(base) != bench.code_only(base.replace('"a // b"', '"a // c"'))
    hashes = {bench.kernel_hash(k) for k in ("topk_rows_kernel<4,4>", "topk_warp_rows_kernel<2>")}
    assert len(hashes) == 2


def test_bench_traffic_table():
    """bench.py reads each workload's measured DRAM traffic from a JSON data file;
    a figure counts only for the kernel (and kernel code) it was measured on."""
    import json

    import bench
    with open(os.path.join(bench.ROOT, bench.TRAFFIC_FILE), encoding="utf-8") as fh:
        table = json.load(fh)
    assert table
    for wl, e in table.items():
        assert {"kernel", "kernel_hash", "dram_bytes_per_launch", "summary"} <= set(e)
        assert os.path.exists(os.path.join(bench.ROOT, e["summary"])), e["summary"]
        t, note = bench.profiled_traffic(wl, e["kernel"])
        if e["kernel_hash"] == bench.kernel_hash(e["kernel"]):
            assert t == e["dram_bytes_per_launch"]
        else:
            assert t is None and note.startswith("stale")
        other = "topk_warp_rows_kernel<4>" if not e["kernel"].startswith("topk_warp_rows") else "topk_rows_kernel<4,4>"
        assert bench.profiled_traffic(wl, other)[0] is None
    assert bench.profiled_traffic("no-such-workload", "topk_rows_kernel<4,4>")[0] is None


def test_bench_sample_rows_bounded():
    import bench
    import workloads
    c4 = workloads.WORKLOADS["c4"]
    rows = bench.sample_rows(c4, 256)
    assert len(rows) == 256 and rows[0] == 0 and rows[-1] < c4.batch and rows == sorted(set(rows))
    assert bench.sample_rows(workloads.WORKLOADS["c2"], 256) == list(range(64))


@pytest.mark.parametrize("temperature,top_p,u,vals,idx,tok,flag,code", [
    (0.0, 0.9, P, P, P, P, P, dstk.EINVAL),            # temperature 0
    (-1.0, 0.9, P, P, P, P, P, dstk.EINVAL),           # negative temperature
    (float("inf"), 0.9, P, P, P, P, P, dstk.EINVAL),   # infinite temperature
    (float("nan"), 0.9, P, P, P, P, P, dstk.EINVAL),   # NaN temperature
    (1.0, 0.0, P, P, P, P, P, dstk.EINVAL),            # top_p 0
    (1.0, 1.5, P, P, P, P, P, dstk.EINVAL),            # top_p above 1
    (1.0, float("nan"), P, P, P, P, P, dstk.EINVAL),   # NaN top_p
    (1.0, 0.9, 0, P, P, P, P, dstk.EINVAL),            # u NULL
    (1.0, 0.9, P, 0, P, P, P, dstk.EINVAL),            # values NULL (required)
    (1.0, 0.9, P, P, 0, P, P, dstk.EINVAL),            # indices NULL
    (1.0, 0.9, P, P, P, 0, P, dstk.EINVAL),            # tokens NULL
    (1.0, 0.9, P, P, P, P, 0, dstk.EINVAL),            # nan_flag NULL
    (1.0, 0.9, P + 2, P, P, P, P, dstk.EALIGN),        # u misaligned
    (1.0, 0.9, P, P, P, P + 2, P, dstk.EALIGN),        # tokens misaligned
    (1.0, 0.9, P, P + 2, P, P, P, dstk.EALIGN),        # fp32 values misaligned
])
def test_sample_argument_errors(temperature, top_p, u, vals, idx, tok, flag, code):
    """ds_topk_sample validates every argument before it enqueues anything (so
    these calls need no GPU): the sampling parameters first, then the sizes,
    pointers and alignments as ds_topk does."""
    assert dstk.ds_topk_sample(P, dstk.FP32, 4, 4096, 4096, 64, temperature, top_p, u, vals, idx, tok,
                               flag, 0) == code


def test_sample_batch_zero_is_ok_without_pointers():
    assert dstk.ds_topk_sample(0, dstk.FP32, 0, 4096, 4096, 64, 1.0, 0.9, 0, 0, 0, 0, 0, 0) == dstk.OK
