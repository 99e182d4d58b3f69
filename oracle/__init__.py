"""CPU oracle for batched row-wise TopK — TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the `cpu_baseline` / `--impl
reference` legs of `bench.py` may import this package. The CUDA library never
imports, links or calls it, and it shares no code with the library: the oracle is
`topk_oracle.c`, a plain sort of (value, index) pairs by the total order
"value descending, index ascending" (see that file's header for the pages it
follows), compiled with gcc into `liboracle_topk.so` beside this file.

Every function here is marshalling around that C routine; there is no selection
arithmetic in Python.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_topk.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math, no -march=native: the shared
    object travels to other hosts). Returns the path of the shared object."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle shared object."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    lib.oracle_topk.restype = ctypes.c_int
    lib.oracle_topk.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_cores.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def cores() -> int:
    return int(load().oracle_cores())


def topk(x: torch.Tensor, k: int, length: Optional[int] = None, return_value: bool = True,
         nthreads: int = 0, lib=None, order: str = "index") -> Tuple[Optional[torch.Tensor], torch.Tensor, int, torch.Tensor]:
    """Oracle TopK of a CPU tensor x [batch, row_stride] (bf16 or fp32).

    Returns (values or None, indices int32 [batch,k], nan_flag int, row_nan bool
    [batch]). order="index": ascending index order; order="value": the total order
    itself (value descending, equal values by ascending index). Rows holding a NaN
    get indices -1.
    """
    if order not in ("index", "value"):
        raise ValueError(order)
    if x.device.type != "cpu":
        raise ValueError("the oracle runs on host memory only")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(x.dtype)
    x = x.contiguous()
    batch, stride = x.shape
    length = stride if length is None else length
    dtype = 0 if x.dtype == torch.bfloat16 else 1
    idx = torch.empty((batch, k), dtype=torch.int32)
    vals = torch.empty((batch, k), dtype=x.dtype) if return_value else None
    flag = np.zeros(1, dtype=np.int32)
    row_nan = np.zeros(max(batch, 1), dtype=np.uint8)
    lib = lib or load()
    rc = lib.oracle_topk(x.data_ptr(), dtype, batch, length, stride, k, 2 if order == "value" else 1,
                         int(return_value),
                         vals.data_ptr() if vals is not None else None, idx.data_ptr(),
                         flag.ctypes.data, row_nan.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_topk failed with code {rc}")
    return vals, idx, int(flag[0]), torch.from_numpy(row_nan[:batch].astype(bool))


def time_topk(x: torch.Tensor, k: int, length: Optional[int] = None, return_value: bool = True,
              nthreads: int = 0, min_seconds: float = 0.0, max_reps: int = 1000) -> Tuple[float, int]:
    """Wall time (s) of one oracle call on x, as the median over repeats that
    together take at least min_seconds. Returns (seconds per call, repeats)."""
    times = []
    t_total = 0.0
    while True:
        t0 = time.perf_counter()
        topk(x, k, length, return_value, nthreads)
        dt = time.perf_counter() - t0
        times.append(dt)
        t_total += dt
        if t_total >= min_seconds or len(times) >= max_reps:
            break
    times.sort()
    return times[len(times) // 2], len(times)
