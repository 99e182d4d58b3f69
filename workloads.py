"""Seeded synthetic inputs for the batched TopK workloads.

This module only draws numbers: it holds none of the selection arithmetic, and
both the CUDA path's tests/benchmark and the CPU oracle's tests take their inputs
from it. Every array is a pure function of (seed, row, column), so any subset of
rows can be regenerated on any device without generating the rest.

Random source: SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom
Number Generators", OOPSLA 2014), used as a counter-based generator: draw n of
stream s is mix64(s + (n + 1) * 0x9E3779B97F4A7C15), where mix64 is SplitMix64's
output function. The counter of element (row, i) is n = row * 2**32 + i.
Normals use the Box-Muller transform in float64 (one cosine branch per element),
then round to float32 (round-to-nearest-even) and, for bf16, float32 -> bf16 (RNE).

Workload shapes follow the pages' examples: the Lightning-Indexer call example
(bf16, 4 x 204800, topk=1024, sorted_index=True, int32 indices) and the two
benchmark groups (bf16 with topk=512; fp32 sampling over vocab 129280 with
topk=512), from the deepseek.csdn.net article "DeepSeek 一次开源三个仓库", section
三 (算子层). The -inf causal tail, the +10 boosted logits and the adversarial rows
are this project's readings of "indexer decode shape", "sampler logits" and
"worst-case scan order"; no public dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterable, Optional, Sequence

import torch

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _s64(u: int) -> int:
    """uint64 constant -> the int64 with the same bits (torch has no full uint64)."""
    u &= _MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 tensors holding uint64 bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def mix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function on int64 tensors (wrapping arithmetic = uint64 bits)."""
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def mix64_int(z: int) -> int:
    """Same function on a Python int (used to check the tensor version)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def draw_int(seed: int, stream: int, n: int) -> int:
    """Draw n (>= 0) of stream `stream` as a Python int in [0, 2**64)."""
    s = (seed * 64 + stream) & _MASK64
    return mix64_int(s + (n + 1) * _GAMMA)


def draws(seed: int, stream: int, rows: torch.Tensor, cols: torch.Tensor) -> torch.Tensor:
    """int64 tensor [len(rows), len(cols)] of draws (uint64 bits) for counters row*2**32+col."""
    s = _s64((seed * 64 + stream) & _MASK64)
    n = rows.to(torch.int64)[:, None] * (1 << 32) + cols.to(torch.int64)[None, :]
    # s + (n + 1) * GAMMA, wrapping
    z = (n + 1) * _s64(_GAMMA) + s
    return mix64(z)


def uniform01(z: torch.Tensor, open_at_zero: bool) -> torch.Tensor:
    """Top 53 bits of a draw -> float64 in [0,1) (or (0,1] when open_at_zero)."""
    top = _lsr(z, 11).to(torch.float64)
    if open_at_zero:
        top = top + 1.0
    return top * (2.0 ** -53)


def normal(seed: int, rows: torch.Tensor, cols: torch.Tensor) -> torch.Tensor:
    """float64 N(0,1) per (row, col) via Box-Muller on streams 0 and 1."""
    u1 = uniform01(draws(seed, 0, rows, cols), open_at_zero=True)
    u2 = uniform01(draws(seed, 1, rows, cols), open_at_zero=False)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def round_to(x64: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """float64 -> float32 (RNE) -> dtype (RNE for bf16)."""
    x32 = x64.to(torch.float32)
    return x32 if dtype == torch.float32 else x32.to(dtype)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    batch: int
    length: int
    k: int
    sorted_index: bool
    return_value: bool
    kind: str
    seed: int
    description: str

    @property
    def elem_size(self) -> int:
        return 2 if self.dtype == torch.bfloat16 else 4

    @property
    def bytes_in(self) -> int:
        return self.batch * self.length * self.elem_size

    @property
    def bytes_out(self) -> int:
        per = 4 + (self.elem_size if self.return_value else 0)
        return self.batch * self.k * per

    def scaled(self, batch: int) -> "Workload":
        return dataclasses.replace(self, batch=batch)


WORKLOADS = {
    "c1": Workload("c1", torch.float32, 4, 4096, 64, False, True, "normal", 20260001,
                   "fp32 TopK, batch 4, row length 4096, k=64, N(0,1), unsorted, values+indices"),
    "c2": Workload("c2", torch.float32, 64, 129280, 512, False, True, "sampler", 20260002,
                   "sampler: fp32 logits, batch 64, vocab 129280, k=512, 3*N(0,1) with 32 "
                   "positions per row boosted by +10, values+indices, unsorted"),
    "c3": Workload("c3", torch.bfloat16, 4, 204800, 1024, True, True, "normal", 20260003,
                   "indexer: bf16, batch 4, row length 204800, k=1024, N(0,1) rounded to bf16, "
                   "sorted_index, values+indices"),
    "c4": Workload("c4", torch.bfloat16, 16384, 32768, 512, False, False, "causal", 20260004,
                   "indexer decode: bf16, batch 16384, row length 32768, k=512, N(0,1) bf16 "
                   "with the last 25% of each row -inf, indices only, unsorted"),
    "c5": Workload("c5", torch.bfloat16, 8, 1048576, 4096, False, True, "adversarial", 20260005,
                   "adversarial: bf16, batch 8, row length 1048576, k=4096, rows cycle "
                   "ascending ramp / 16 levels / sorted N(0,1), values+indices, unsorted"),
}

# Stream tags inside one seed.
_STREAM_BOOST = 2
_STREAM_LEVEL = 3


def _rows_tensor(rows: Iterable[int] | torch.Tensor, device) -> torch.Tensor:
    if isinstance(rows, torch.Tensor):
        return rows.to(device=device, dtype=torch.int64)
    return torch.tensor(list(rows), dtype=torch.int64, device=device)


def generate_rows(w: Workload, rows: Sequence[int] | torch.Tensor, device="cpu",
                  row_stride: Optional[int] = None, pad_value: float = float("nan"),
                  chunk_rows: int = 512) -> torch.Tensor:
    """Rows `rows` of workload `w` as a [len(rows), row_stride] tensor of w.dtype.

    Columns [length, row_stride) hold `pad_value` (NaN by default, so a path that
    reads padding is caught by the NaN flag).
    """
    rows_t = _rows_tensor(rows, device)
    stride = w.length if row_stride is None else row_stride
    out = torch.empty((rows_t.numel(), stride), dtype=w.dtype, device=device)
    if stride > w.length:
        out[:, w.length:] = pad_value
    cols = torch.arange(w.length, dtype=torch.int64, device=device)
    for r0 in range(0, rows_t.numel(), chunk_rows):
        rr = rows_t[r0:r0 + chunk_rows]
        out[r0:r0 + rr.numel(), :w.length] = _gen_block(w, rr, cols)
    return out


def generate(w: Workload, device="cpu", row_stride: Optional[int] = None,
             pad_value: float = float("nan")) -> torch.Tensor:
    """The whole batch of workload w."""
    return generate_rows(w, range(w.batch), device, row_stride, pad_value)


def _gen_block(w: Workload, rows: torch.Tensor, cols: torch.Tensor) -> torch.Tensor:
    L = w.length
    if w.kind == "normal":
        return round_to(normal(w.seed, rows, cols), w.dtype)
    if w.kind == "sampler":
        x = 3.0 * normal(w.seed, rows, cols)
        # 32 distinct boosted positions per row: the 32 columns with the smallest
        # draws of the boost stream (a uniformly random 32-subset).
        keys = draws(w.seed, _STREAM_BOOST, rows, cols)
        # order by unsigned value: flip the sign bit so signed order = unsigned order
        keys = keys ^ _s64(1 << 63)
        pos = torch.argsort(keys, dim=1, stable=True)[:, :32]
        x.scatter_add_(1, pos, torch.full(pos.shape, 10.0, dtype=x.dtype, device=x.device))
        return round_to(x, w.dtype)
    if w.kind == "causal":
        x = round_to(normal(w.seed, rows, cols), w.dtype)
        x[:, (3 * L) // 4:] = float("-inf")
        return x
    if w.kind == "adversarial":
        out = torch.empty((rows.numel(), L), dtype=w.dtype, device=rows.device)
        kinds = rows % 3
        for kind in (0, 1, 2):
            sel = (kinds == kind).nonzero().flatten()
            if sel.numel() == 0:
                continue
            rsel = rows[sel]
            if kind == 0:    # non-decreasing ramp with bf16 plateaus (ties)
                ramp = -4.0 + 8.0 * cols.to(torch.float64) / L
                blk = round_to(ramp, w.dtype)[None, :].expand(rsel.numel(), L)
            elif kind == 1:  # 16 levels (j - 8) / 2, j uniform in 0..15
                j = _lsr(draws(w.seed, _STREAM_LEVEL, rsel, cols), 60).to(torch.float64)
                blk = round_to((j - 8.0) / 2.0, w.dtype)
            else:            # N(0,1) -> bf16, then sorted ascending
                blk = round_to(normal(w.seed, rsel, cols), w.dtype)
                blk = torch.sort(blk.to(torch.float32), dim=1, stable=True).values.to(w.dtype)
            out[sel] = blk
        return out
    raise ValueError(f"unknown workload kind {w.kind!r}")


def random_rows(batch: int, length: int, dtype: torch.dtype, seed: int, style: str = "normal",
                device="cpu", row_stride: Optional[int] = None) -> torch.Tensor:
    """Ad-hoc seeded rows for sweeps and edge cases.

    style: 'normal' N(0,1); 'ties' 4 levels {-1, 0, 1, 2}; 'allequal' all 1.0;
    'ramp' strictly increasing ints (exact in fp32; bf16 rounds it into plateaus);
    'signed_zero' random mix of +0.0 / -0.0 / 1.0 / -inf / +inf;
    'denormal' tiny magnitudes around the smallest subnormal, both signs.
    """
    rows = torch.arange(batch, dtype=torch.int64, device=device)
    cols = torch.arange(length, dtype=torch.int64, device=device)
    stride = length if row_stride is None else row_stride
    if style == "normal":
        x = round_to(normal(seed, rows, cols), dtype)
    elif style == "ties":
        j = _lsr(draws(seed, _STREAM_LEVEL, rows, cols), 62).to(torch.float64)
        x = round_to(j - 1.0, dtype)
    elif style == "allequal":
        x = torch.ones((batch, length), dtype=dtype, device=device)
    elif style == "ramp":
        x = round_to(cols.to(torch.float64)[None, :].expand(batch, length).clone(), dtype)
    elif style == "signed_zero":
        j = _lsr(draws(seed, _STREAM_LEVEL, rows, cols), 61)
        table = torch.tensor([0.0, -0.0, 1.0, float("-inf"), float("inf"), -0.0, 0.0, 1.0],
                             dtype=torch.float64, device=device)
        x = round_to(table[j], dtype)
    elif style == "denormal":
        j = _lsr(draws(seed, _STREAM_LEVEL, rows, cols), 60).to(torch.float64)  # 0..15
        tiny = 2.0 ** -149 if dtype == torch.float32 else 2.0 ** -133
        x = round_to((j - 8.0) * tiny, dtype)
    else:
        raise ValueError(style)
    if stride == length:
        return x.contiguous()
    out = torch.full((batch, stride), float("nan"), dtype=dtype, device=device)
    out[:, :length] = x
    return out
