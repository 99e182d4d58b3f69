"""Oracle of the sampler tail: top-k -> temperature softmax -> top-p -> one draw.

TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the benchmark's
CPU-baseline leg may use it; the product path never does.

What it computes, per row, in float64 (the steps in the order the sampler takes
them; deepseek.csdn.net, "DeepSeek 一次开源三个仓库": the request's temperature and
top_p; github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点:
the sampler path of TopK picks the next token among the k largest logits):
  1. the k selected pairs in value order (value descending, equal values by
     ascending index), from the TopK oracle;
  2. weights w_j = exp((v_j - v_0) / T), v_0 the largest value (w_0 = 1);
     when v_0 is +inf the elements equal to +inf weigh 1 and the rest 0;
  3. cumulative sums C_j = w_0 + ... + w_j and W = C_{k-1}; the nucleus is the
     shortest prefix [0, m] with C_m >= top_p * W;
  4. with u in [0, 1), the token is the element at the first j <= m with
     C_j > u * C_m.
Readings where the pages are silent: probabilities over the k survivors only
(softmax after the cut to k); top-p keeps the shortest prefix reaching the mass
(>=); the draw uses the inverse CDF with a strict > so that u = 0 picks the
largest value; the uniform number is an input, not drawn inside.
"""
from typing import Tuple

import numpy as np
import torch

from . import topk as _topk


def weights(v: np.ndarray, temperature: float) -> np.ndarray:
    """Step 2 on one row of k values (value order), float64."""
    v = v.astype(np.float64)
    v0 = v[0]
    if np.isposinf(v0):
        return (v == v0).astype(np.float64)
    if np.isneginf(v0):  # every value is -inf: the first (lowest index) takes all
        w = np.zeros_like(v)
        w[0] = 1.0
        return w
    return np.exp((v - v0) / temperature)


def draw(w: np.ndarray, top_p: float, u: float) -> Tuple[int, int]:
    """Steps 3-4 on one row's weights: (position of the token, nucleus size)."""
    c = np.cumsum(w)
    total = c[-1]
    m = int(np.argmax(c >= top_p * total))  # first prefix end reaching the mass
    target = u * c[m]
    j = int(np.argmax(c[: m + 1] > target))
    return j, m + 1


def sample(x: torch.Tensor, k: int, temperature: float, top_p: float, u: np.ndarray
           ) -> Tuple[np.ndarray, np.ndarray, torch.Tensor, torch.Tensor, np.ndarray]:
    """Sampler oracle on a CPU tensor x [batch, len] (bf16 or fp32).

    Returns (tokens int64 [batch], positions in value order [batch], top-k
    indices [batch, k] in value order, top-k values [batch, k], row_nan [batch]).
    Rows holding a NaN get token -1.
    """
    vals, idx, _, row_nan = _topk(x, k, return_value=True, order="value")
    vf = vals.to(torch.float64).numpy()
    tokens = np.full(x.shape[0], -1, dtype=np.int64)
    pos = np.full(x.shape[0], -1, dtype=np.int64)
    for b in range(x.shape[0]):
        if bool(row_nan[b]):
            continue
        j, _ = draw(weights(vf[b], temperature), top_p, float(u[b]))
        pos[b] = j
        tokens[b] = int(idx[b, j])
    return tokens, pos, idx, vals, row_nan.numpy()
