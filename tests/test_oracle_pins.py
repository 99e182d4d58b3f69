"""Pins of the CPU oracle against things other than itself (CPU only).

- hand-worked golden cases (tests/golden/*.txt, derived from the definition);
- the brute-force O(n^2) rank definition on tiny rows, all k, adversarial values;
- exhaustive enumeration of short rows over small alphabets with +-0 and +-inf;
- the invariants every TopK result has, on rows shaped like each workload;
- torch.topk on tie-free rows (values as a multiset, index sets when distinct);
- closed forms on structured rows (all-equal, strictly increasing, 16-level, -inf tail);
- the NaN flag (never set by padding);
- planted mistakes: mutated copies of the oracle source must fail these pins.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import (as_f64, bits_of, brute_force_selected, check_invariants, load_golden,
                         tensor_from_bits)

DTYPES = [torch.float32, torch.bfloat16]


def _golden_check(lib, fname, dtype):
    failures = []
    for case in load_golden(fname, dtype):
        n_x = len(case["x"])
        length = case.get("len", n_x)
        x = tensor_from_bits(case["x"], dtype).reshape(1, n_x)
        vals, idx, flag, row_nan = oracle.topk(x, case["k"], length=length, lib=lib)
        if (flag & 1) != case["nan"]:
            failures.append((case["name"], "nan flag", flag))
            continue
        if case["nan"]:
            continue
        if idx[0].tolist() != case["indices"]:
            failures.append((case["name"], "indices", idx[0].tolist(), case["indices"]))
        if bits_of(vals[0]).tolist() != case["values"]:
            failures.append((case["name"], "values", bits_of(vals[0]).tolist(), case["values"]))
    return failures


def test_generator_matches_definition():
    """The vectorised SplitMix64 draws equal the scalar definition."""
    rows = torch.tensor([0, 1, 7, 123456], dtype=torch.int64)
    cols = torch.tensor([0, 1, 2, 4095, 2**31 - 1], dtype=torch.int64)
    z = workloads.draws(42, 3, rows, cols)
    for a, r in enumerate(rows.tolist()):
        for b, c in enumerate(cols.tolist()):
            want = workloads.draw_int(42, 3, r * 2**32 + c)
            assert (z[a, b].item() & (2**64 - 1)) == want


def test_generator_distributions():
    """Sanity of the workload recipes (shape, dtype, -inf tail, boosts, levels)."""
    w4 = workloads.WORKLOADS["c4"]
    x4 = workloads.generate_rows(w4, [0, 5])
    assert x4.dtype == torch.bfloat16 and x4.shape == (2, 32768)
    assert torch.isinf(x4[:, 24576:]).all() and (x4[:, 24576:] < 0).all()
    assert torch.isfinite(x4[:, :24576]).all()
    z = x4[:, :24576].float()
    assert abs(z.mean().item()) < 0.05 and abs(z.std().item() - 1) < 0.05
    w2 = workloads.WORKLOADS["c2"]
    x2 = workloads.generate_rows(w2, [3])
    assert (x2 > 9.0).sum().item() >= 28   # 32 boosted logits sit near +10
    w5 = workloads.WORKLOADS["c5"]
    x5 = workloads.generate_rows(w5, [0, 1, 2])
    assert torch.all(x5[0, 1:].float() >= x5[0, :-1].float())
    assert torch.unique(x5[1].float()).numel() == 16
    assert torch.all(x5[2, 1:].float() >= x5[2, :-1].float())


@pytest.mark.parametrize("fname,dtype", [("handworked_fp32.txt", torch.float32),
                                         ("handworked_bf16.txt", torch.bfloat16)])
def test_golden_handworked(fname, dtype):
    assert _golden_check(oracle.load(), fname, dtype) == []


def _bruteforce_check(lib, dtype, styles=("normal", "ties", "signed_zero", "denormal", "allequal"),
                      lengths=(1, 2, 3, 5, 8, 13, 31, 64), seed=7):
    bad = []
    for style in styles:
        for n in lengths:
            x = workloads.random_rows(6, n, dtype, seed + n, style=style)
            want = brute_force_selected(as_f64(x), 1)  # warm shape
            for k in range(1, n + 1):
                vals, idx, flag, _ = oracle.topk(x, k, lib=lib)
                want = brute_force_selected(as_f64(x), k)
                for b in range(x.shape[0]):
                    got = np.zeros(n, dtype=bool)
                    got[idx[b].numpy()] = True
                    if not np.array_equal(got, want[b]) or not np.all(np.diff(idx[b].numpy()) > 0):
                        bad.append((style, n, k, b))
                    elif not np.array_equal(bits_of(vals[b]), bits_of(x[b])[idx[b].numpy()]):
                        bad.append((style, n, k, b, "values"))
    return bad


@pytest.mark.parametrize("dtype", DTYPES)
def test_bruteforce_tiny_rows(dtype):
    assert _bruteforce_check(oracle.load(), dtype) == []


def _exhaustive_check(lib, dtype, max_len=5):
    alphabet = [float("-inf"), -1.0, -0.0, 0.0, 1.0, float("inf")]
    bad = []
    for n in range(1, max_len + 1):
        rows = np.array(list(itertools.product(alphabet, repeat=n)), dtype=np.float64)
        x = torch.tensor(rows, dtype=torch.float64).to(dtype)
        for k in range(1, n + 1):
            vals, idx, flag, _ = oracle.topk(x, k, lib=lib)
            want = brute_force_selected(as_f64(x), k)
            got = np.zeros_like(want)
            np.put_along_axis(got, idx.numpy().astype(np.int64), True, axis=1)
            if not np.array_equal(got, want):
                bad.append((n, k, int((got != want).any(axis=1).sum())))
            if not np.array_equal(bits_of(vals), np.take_along_axis(bits_of(x), idx.numpy().astype(np.int64), 1)):
                bad.append((n, k, "values"))
    return bad


@pytest.mark.parametrize("dtype", DTYPES)
def test_exhaustive_small_alphabet(dtype):
    assert _exhaustive_check(oracle.load(), dtype) == []


def _sample_rows(name):
    w = workloads.WORKLOADS[name]
    rows = {"c1": [0, 1, 2, 3], "c2": [0, 31, 63], "c3": [1], "c4": [0, 9999], "c5": [0, 1, 2]}[name]
    return w, workloads.generate_rows(w, rows)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_invariants_on_workload_rows(name):
    w, x = _sample_rows(name)
    vals, idx, flag, row_nan = oracle.topk(x, w.k)
    assert flag == 0 and not row_nan.any()
    for b in range(x.shape[0]):
        check_invariants(x[b], w.k, idx[b].numpy(), bits_of(vals[b]))


def test_torch_topk_on_tie_free_rows():
    """Where no tie sits at the k-th value, the selected values equal torch.topk's
    as a multiset; with all values distinct the index sets match too."""
    x = workloads.random_rows(16, 4096, torch.float32, 99, style="normal")
    for k in (1, 64, 1000, 4096):
        vals, idx, _, _ = oracle.topk(x, k)
        tv, ti = torch.topk(x, k, dim=1)
        for b in range(x.shape[0]):
            row = x[b]
            kth = tv[b, -1]
            if (row == kth).sum().item() != 1:
                continue  # a tie at the k-th value: torch's choice is arbitrary
            assert torch.equal(torch.sort(vals[b]).values, torch.sort(tv[b]).values)
            if torch.unique(row).numel() == row.numel():
                assert set(idx[b].tolist()) == set(ti[b].tolist())


def test_closed_forms():
    # all equal -> the k lowest indices
    x = workloads.random_rows(2, 1000, torch.bfloat16, 1, style="allequal")
    _, idx, _, _ = oracle.topk(x, 77)
    assert idx[0].tolist() == list(range(77))
    # strictly increasing fp32 ramp -> the last k indices
    x = workloads.random_rows(1, 5000, torch.float32, 1, style="ramp")
    _, idx, _, _ = oracle.topk(x, 300)
    assert idx[0].tolist() == list(range(4700, 5000))
    # 16-level row: all k from the top level present, at its k lowest indices
    w5 = workloads.WORKLOADS["c5"]
    x = workloads.generate_rows(w5, [1])
    v = as_f64(x)[0]
    top = v.max()
    where = np.nonzero(v == top)[0]
    assert where.size >= w5.k
    _, idx, _, _ = oracle.topk(x, w5.k)
    assert idx[0].tolist() == where[:w5.k].tolist()
    # causal row: nothing from the -inf tail while k <= #finite
    w4 = workloads.WORKLOADS["c4"]
    x = workloads.generate_rows(w4, [3])
    _, idx, _, _ = oracle.topk(x, w4.k)
    assert idx.max().item() < 24576
    # a -inf tail is selected only once the finite part is exhausted (k > #finite)
    xs = torch.tensor([[2.0, float("-inf"), 1.0, float("-inf"), float("-inf")]])
    _, idx, _, _ = oracle.topk(xs, 4)
    assert idx[0].tolist() == [0, 1, 2, 3]


@pytest.mark.parametrize("dtype", DTYPES)
def test_nan_flag(dtype):
    L = 4096
    base = workloads.random_rows(6, L, dtype, 5, style="normal")
    x = base.clone()
    x[0, 0] = float("nan")
    x[1, L // 2] = float("nan")
    x[2, L - 1] = float("nan")
    x[3, :] = float("-inf")
    x[3, 100] = float("nan")          # NaN inside an all -inf row
    x[4, 7] = -float("nan")            # negative NaN (sign bit set)
    vals, idx, flag, row_nan = oracle.topk(x, 64)
    assert flag == 1
    assert row_nan.tolist() == [True, True, True, True, True, False]
    # the clean row is still exact
    _, idx_clean, _, _ = oracle.topk(base[5:6], 64)
    assert torch.equal(idx[5], idx_clean[0])
    # padding NaN is never read
    xp = workloads.random_rows(3, 100, dtype, 6, style="normal", row_stride=128)
    assert torch.isnan(xp[:, 100:]).all()
    _, _, flag, _ = oracle.topk(xp, 10, length=100)
    assert flag == 0


# ---- planted mistakes --------------------------------------------------------------

_MUTANTS = {
    "tie_break_reversed": ("if (a->index < b->index) return -1;\n  if (a->index > b->index) return 1;",
                           "if (a->index < b->index) return 1;\n  if (a->index > b->index) return -1;"),
    "ascending_values": ("if (a->value > b->value) return -1;\n  if (a->value < b->value) return 1;",
                         "if (a->value > b->value) return 1;\n  if (a->value < b->value) return -1;"),
    "values_from_rank_not_index": ("memcpy(ov, row + (size_t)pairs[j].index * esize, esize);",
                                   "memcpy(ov, row + (size_t)j * esize, esize);"),
    "nan_check_dropped": ("if (isnan(pairs[i].value)) has_nan = 1;", ";"),
    "bf16_decoded_low_half": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h;"),
    "last_pair_dropped": ("qsort(pairs, (size_t)job->k, sizeof(oracle_pair), by_index_asc);",
                          "qsort(pairs, (size_t)job->k - 1, sizeof(oracle_pair), by_index_asc);"),
    # -0.0 ordered below +0.0 (what a raw-bit comparison would do)
    "signed_zero_by_bits": ("if (a->value < b->value) return 1;\n",
                            "if (a->value < b->value) return 1;\n  if (signbit(a->value) != "
                            "signbit(b->value)) return signbit(a->value) ? 1 : -1;\n"),
}


def _all_pins_pass(lib) -> bool:
    try:
        if _golden_check(lib, "handworked_fp32.txt", torch.float32):
            return False
        if _golden_check(lib, "handworked_bf16.txt", torch.bfloat16):
            return False
        for dt in DTYPES:
            if _exhaustive_check(lib, dt, max_len=4):
                return False
            if _bruteforce_check(lib, dt, lengths=(5, 13), styles=("ties", "normal")):
                return False
        return True
    except (AssertionError, RuntimeError, ValueError, IndexError):
        return False


@pytest.mark.parametrize("mutant", sorted(_MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path):
    """Each plausible mistake, planted in a temporary copy of the oracle, fails a pin."""
    old, new = _MUTANTS[mutant]
    src = open(oracle._SRC, encoding="utf-8").read()
    assert old in src, f"mutation site for {mutant} not found"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new), encoding="utf-8")
    so = oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    assert not _all_pins_pass(lib), f"planted mistake {mutant} passed every pin"


def test_unmutated_oracle_passes_pin_subset():
    assert _all_pins_pass(oracle.load())


# ---- value order (sorted_index = 2) ----------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("style", ["normal", "ties", "signed_zero", "denormal", "ramp"])
def test_value_order_matches_stable_sort(dtype, style):
    """Value order is the first k pairs of a stable descending sort: values
    descending, equal values (including -0.0 and +0.0) by ascending index."""
    x = workloads.random_rows(5, 333, dtype, 4711, style=style)
    for k in (1, 7, 100, 333):
        v, i, f, rn = oracle.topk(x, k, order="value")
        assert f == 0
        ref = torch.sort(x.to(torch.float64), dim=1, descending=True, stable=True)
        assert torch.equal(i.to(torch.int64), ref.indices[:, :k])
        assert np.array_equal(bits_of(v), bits_of(torch.gather(x, 1, i.to(torch.int64))))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_value_order_same_set_as_index_order(dtype):
    x = workloads.random_rows(4, 2000, dtype, 99, style="normal")
    x[1, 100:400] = 1.0  # a long run of equal values across the k-th position
    for k in (64, 350, 2000):
        vv, iv, _, _ = oracle.topk(x, k, order="value")
        vi, ii, _, _ = oracle.topk(x, k, order="index")
        assert torch.equal(torch.sort(iv, dim=1).values, ii)
        keys = vv.to(torch.float64)
        assert bool((keys[:, 1:] <= keys[:, :-1]).all())  # non-increasing values
