"""Test helpers: golden-file parsing, a brute-force rank definition of TopK, and
the invariant checker applied to every oracle and GPU result. Independent of the
oracle's C code and of the CUDA library."""
from __future__ import annotations

import os
import struct
from typing import Dict, List, Optional

import numpy as np
import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(tok: str, dtype: torch.dtype) -> int:
    if tok.lower().startswith("0x"):
        return int(tok, 16)
    f = float(tok)
    b32 = struct.unpack("<I", struct.pack("<f", f))[0]
    if dtype == torch.float32:
        return b32
    if f != f:
        return 0x7FC0
    if (b32 & 0xFFFF) != 0:
        raise ValueError(f"{tok} is not exact in bf16")
    return b32 >> 16


def tensor_from_bits(bits: List[int], dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.float32:
        return torch.tensor(np.array(bits, dtype=np.uint32).view(np.int32)).view(torch.float32)
    return torch.tensor(np.array(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def load_golden(name: str, dtype: torch.dtype) -> List[Dict]:
    cases, cur = [], None
    with open(os.path.join(GOLDEN_DIR, name), encoding="utf-8") as fh:
        for raw in fh:
            line = raw.strip()
            if line.startswith("#"):
                continue
            if not line:
                if cur:
                    cases.append(cur)
                cur = None
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
            elif key in ("k", "len", "nan"):
                cur[key] = int(rest)
            elif key in ("x", "values"):
                cur[key] = [_bits(t, dtype) for t in rest.split()]
            elif key == "indices":
                cur[key] = [int(t) for t in rest.split()]
            else:
                raise ValueError(f"bad golden line {line!r}")
    if cur:
        cases.append(cur)
    return cases


def as_f64(x: torch.Tensor) -> np.ndarray:
    """Exact float64 copy (torch's own bf16/fp32 -> float64 conversion)."""
    return x.detach().cpu().to(torch.float64).numpy()


def brute_force_selected(v: np.ndarray, k: int) -> np.ndarray:
    """Boolean mask [B, n] of the k selected columns per row, by the rank
    definition: column i is selected iff fewer than k columns precede it in the
    total order, i.e. #{j: v_j > v_i} + #{j < i: v_j == v_i} < k. O(n^2)."""
    B, n = v.shape
    gt = (v[:, None, :] > v[:, :, None]).sum(axis=2)            # [B, i] count of j with v_j > v_i
    eq = (v[:, None, :] == v[:, :, None])                       # [B, i, j]
    lower = np.tril(np.ones((n, n), dtype=bool), k=-1)          # j < i
    eq_before = (eq & lower[None]).sum(axis=2)
    return (gt + eq_before) < k


def check_invariants(x_row: torch.Tensor, k: int, idx: np.ndarray, vals_bits: Optional[np.ndarray],
                     require_sorted: bool = True) -> None:
    """Assert every property a correct TopK result of one NaN-free row has."""
    n = x_row.numel()
    v = as_f64(x_row)
    idx = np.asarray(idx, dtype=np.int64)
    assert idx.shape == (k,), idx.shape
    assert idx.min() >= 0 and idx.max() < n, "index out of range"
    if require_sorted:
        assert np.all(np.diff(idx) > 0), "indices not strictly ascending"
    else:
        idx = np.sort(idx)
        assert np.all(np.diff(idx) > 0), "duplicate indices"
    if vals_bits is not None:
        assert np.array_equal(np.asarray(vals_bits), bits_of(x_row)[idx]), "values are not x[idx]"
    sel = np.zeros(n, dtype=bool)
    sel[idx] = True
    vk = v[idx].min()
    assert (v > vk).sum() < k <= (v >= vk).sum(), "count invariant violated"
    assert np.all(v[~sel] <= vk), "an unselected value exceeds the k-th value"
    ties = np.nonzero(v == vk)[0]
    n_tie_sel = sel[ties].sum()
    assert np.all(sel[ties[:n_tie_sel]]) and not np.any(sel[ties[n_tie_sel:]]), \
        "ties at the k-th value not resolved to the lowest indices"
