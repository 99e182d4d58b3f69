"""Pins of the sampler-tail oracle (oracle/sampler.py), CPU only, plus the C
entry point's argument checks (which return before touching a GPU)."""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
import oracle.sampler as osam
import workloads


def test_hand_worked_nucleus():
    """v = (2, 1, 0), T = 1: p = (0.665, 0.245, 0.090). top_p = 0.7 keeps the
    first two (0.665 < 0.7 <= 0.910); renormalised they split at 0.731."""
    w = osam.weights(np.array([2.0, 1.0, 0.0]), 1.0)
    p = w / w.sum()
    assert np.allclose(p, [0.66524096, 0.24472847, 0.09003057])
    assert osam.draw(w, 0.7, 0.72) == (0, 2)
    assert osam.draw(w, 0.7, 0.74) == (1, 2)
    assert osam.draw(w, 1.0, 0.95) == (2, 3)
    assert osam.draw(w, 0.6, 0.99) == (0, 1)  # 0.665 >= 0.6: the nucleus is the argmax


@pytest.mark.parametrize("temperature", [0.5, 1.0, 3.0])
def test_draw_matches_scipy_softmax_cdf(temperature):
    """With top_p = 1 the draw is the inverse CDF of softmax(v / T): compare with
    scipy's softmax and numpy's searchsorted on a grid of u."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        v = np.sort(rng.normal(0, 2, size=40))[::-1]
        w = osam.weights(v, temperature)
        cdf = np.cumsum(scipy.special.softmax(v / temperature))
        for u in np.linspace(0, 0.999, 97):
            j, _ = osam.draw(w, 1.0, u)
            ref = int(np.searchsorted(cdf, u, side="right"))
            if j != ref:  # only where u sits on a step, to rounding
                assert abs(cdf[min(j, ref)] - u) < 1e-12


def test_closed_forms():
    v = np.array([3.0, 2.5, 2.5, -1.0])
    for u in (0.0, 0.5, 0.999):
        assert osam.draw(osam.weights(v[:1], 1.0), 1.0, u)[0] == 0  # k = 1: argmax
        assert osam.draw(osam.weights(v, 1.0), 1e-9, u)[0] == 0     # tiny top_p: argmax
    eq = np.zeros(8)
    for i in range(8):  # equal logits: uniform over the k
        assert osam.draw(osam.weights(eq, 1.0), 1.0, (i + 0.5) / 8)[0] == i
    w = osam.weights(np.array([1.0, 0.0]), 1e6)  # huge temperature: nearly uniform
    assert abs(w[1] / w.sum() - 0.5) < 1e-6
    inf = osam.weights(np.array([np.inf, np.inf, 5.0]), 1.0)
    assert list(inf) == [1.0, 1.0, 0.0]
    ninf = osam.weights(np.array([-np.inf, -np.inf]), 1.0)
    assert list(ninf) == [1.0, 0.0]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sample_rows_follow_value_order(dtype):
    """The token is an element of the value-ordered top-k at the drawn position,
    and u -> 0 picks the row's largest value (lowest index among equals)."""
    x = workloads.random_rows(6, 500, dtype, 11, style="ties")
    u0 = np.zeros(6)
    tok, pos, idx, vals, rn = osam.sample(x, 50, 1.0, 1.0, u0)
    assert (pos == 0).all()
    _, top1, _, _ = oracle.topk(x, 1)
    assert np.array_equal(tok, top1[:, 0].numpy())
    u = np.linspace(0.05, 0.95, 6)
    tok, pos, idx, vals, rn = osam.sample(x, 50, 0.7, 0.9, u)
    assert np.array_equal(tok, idx.numpy()[np.arange(6), pos])


def test_entry_point_argument_checks():
    import sampler_topk_selection_ds_b300 as dstk
    P = 1 << 20  # a fake, 16-byte aligned device address: never dereferenced
    ok_args = dict(x=P, dtype=dstk.FP32, batch=2, length=16, row_stride=16, k=4, temperature=1.0,
                   top_p=0.9, u=P, out_values=P, out_indices=P, out_tokens=P, nan_flag=P)
    for bad in (dict(temperature=0.0), dict(temperature=-1.0), dict(temperature=float("inf")),
                dict(temperature=float("nan")), dict(top_p=0.0), dict(top_p=1.5),
                dict(top_p=float("nan")), dict(u=0), dict(out_tokens=0), dict(out_values=0),
                dict(k=0), dict(k=17)):
        a = dict(ok_args, **bad)
        assert dstk.ds_topk_sample(**a) == dstk.EINVAL, bad
    assert dstk.ds_topk_sample(**dict(ok_args, u=P + 2)) == dstk.EALIGN
    assert dstk.ds_topk_sample(**dict(ok_args, batch=0, x=0, u=0, out_values=0, out_indices=0,
                                      out_tokens=0, nan_flag=0)) == dstk.OK
