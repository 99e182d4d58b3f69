"""ctypes binding of libds_topk.so — argument marshalling only.

`ds_topk` mirrors the C entry point one to one (raw integers for pointers and
the stream). `topk` is the tensor-level convenience a PyTorch caller uses: it
allocates the outputs with torch on x's device, then makes the single C call.
No step of the selection runs in Python; if the shared object is missing the
import fails loudly (there is no CPU fallback).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libds_topk.so")

BF16 = 0
FP32 = 1
OK, EINVAL, EALIGN, ECUDA, ETIMEOUT = 0, 1, 2, 3, 4
FLAG_NAN = 1
FLAG_TIMEOUT = 2
MAX_K = 4096
PATH_ROW = 0
PATH_CLUSTER = 1
PATH_WARP_ROWS = 2
INDEX_INT32 = 0
INDEX_INT64 = 1
SORT_NONE = 0   # output order unspecified
SORT_INDEX = 1  # ascending index
SORT_VALUE = 2  # value descending, equal values by ascending index


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("threads_per_cta", ctypes.c_int32), ("vectors_per_granule", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int64), ("granules_per_cta", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int32), ("launches", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class DsTopkError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"ds_topk failed: {status_string(code)} (code {code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m sampler_topk_selection_ds_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.ds_topk.restype = ctypes.c_int
    lib.ds_topk.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.ds_topk_ex.restype = ctypes.c_int
    lib.ds_topk_ex.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                               ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.ds_topk_sample.restype = ctypes.c_int
    lib.ds_topk_sample.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]
    lib.ds_topk_plan.restype = ctypes.c_int
    lib.ds_topk_plan.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(Plan)]
    lib.ds_topk_status_string.restype = ctypes.c_char_p
    lib.ds_topk_status_string.argtypes = [ctypes.c_int]
    lib.ds_topk_version.restype = ctypes.c_int
    lib.ds_topk_version.argtypes = []
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.ds_topk_status_string(code).decode()


def version() -> int:
    return int(lib.ds_topk_version())


def ds_topk(x: int, dtype: int, batch: int, length: int, row_stride: int, k: int,
            sorted_index: int, return_value: int, out_values: Optional[int], out_indices: int,
            nan_flag: int, stream: int = 0) -> int:
    """The C call, verbatim: pointers and the stream are plain integers."""
    return int(lib.ds_topk(x, dtype, batch, length, row_stride, k, sorted_index, return_value,
                           out_values, out_indices, nan_flag, stream))


def ds_topk_ex(x: int, dtype: int, batch: int, length: int, row_stride: int, k: int,
               sorted_index: int, return_value: int, index_type: int, out_values: Optional[int],
               out_indices: int, nan_flag: int, stream: int = 0) -> int:
    """The C call, verbatim: pointers and the stream are plain integers."""
    return int(lib.ds_topk_ex(x, dtype, batch, length, row_stride, k, sorted_index, return_value,
                              index_type, out_values, out_indices, nan_flag, stream))


def ds_topk_sample(x: int, dtype: int, batch: int, length: int, row_stride: int, k: int,
                   temperature: float, top_p: float, u: int, out_values: int, out_indices: int,
                   out_tokens: int, nan_flag: int, stream: int = 0) -> int:
    """The C call, verbatim: pointers and the stream are plain integers."""
    return int(lib.ds_topk_sample(x, dtype, batch, length, row_stride, k, temperature, top_p, u,
                                  out_values, out_indices, out_tokens, nan_flag, stream))


def ds_topk_plan(dtype: int, batch: int, length: int, row_stride: int, k: int,
                 sm_count: int) -> Tuple[int, Plan]:
    plan = Plan()
    rc = int(lib.ds_topk_plan(dtype, batch, length, row_stride, k, sm_count, ctypes.byref(plan)))
    return rc, plan


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return FP32
    raise TypeError(f"ds_topk supports bfloat16 and float32 inputs, not {dt}")


def _order_code(sorted_index) -> int:
    if isinstance(sorted_index, str):
        return {"none": SORT_NONE, "index": SORT_INDEX, "value": SORT_VALUE}[sorted_index]
    if isinstance(sorted_index, bool):
        return SORT_INDEX if sorted_index else SORT_NONE
    return int(sorted_index)


def topk(x: torch.Tensor, k: int, sorted_index=False, return_value: bool = True,
         length: Optional[int] = None, nan_flag: Optional[torch.Tensor] = None,
         out: Optional[Tuple[Optional[torch.Tensor], torch.Tensor]] = None,
         stream: Optional[torch.cuda.Stream] = None, index_dtype: torch.dtype = torch.int32):
    """TopK of each row of a CUDA tensor x [batch, row_stride] (row stride may
    exceed `length`, the number of valid columns; padding is never selected nor
    checked for NaN). Rows need not start on 16-byte boundaries (an offset view,
    or a row stride that is not a multiple of 16 bytes): every kernel reads a row
    as the 16-byte blocks that overlap it and masks the elements outside it.

    sorted_index: False/True (unspecified / ascending index), or "value"
    (SORT_VALUE: value descending, equal values by ascending index).
    index_dtype: torch.int32 (ds_topk) or torch.int64 (ds_topk_ex, INDEX_INT64).
    Returns (values or None, indices [batch, k]). If nan_flag (an int32
    CUDA tensor with one element) is given, DS_TOPK_FLAG_NAN is OR-ed into it
    when a row holds a NaN; the caller clears it.
    """
    if x.dim() != 2:
        raise ValueError("x must be 2-D [batch, row_stride]")
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("rows of x must be contiguous")
    batch = x.shape[0]
    length = x.shape[1] if length is None else int(length)
    row_stride = x.stride(0) if batch > 1 else max(x.shape[1], length)
    if batch <= 1:
        # a single row has no meaningful stride: any multiple of 16 bytes >= length works
        es = x.element_size()
        row_stride = -(-max(length, 1) * es // 16) * 16 // es
    if out is None:
        idx = torch.empty((batch, k), dtype=index_dtype, device=x.device)
        vals = torch.empty((batch, k), dtype=x.dtype, device=x.device) if return_value else None
    else:
        vals, idx = out
    flag = nan_flag if nan_flag is not None else torch.zeros(1, dtype=torch.int32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    if index_dtype not in (torch.int32, torch.int64) or idx.dtype != index_dtype:
        raise ValueError("indices are int32 or int64, matching index_dtype")
    rc = ds_topk_ex(x.data_ptr(), dtype_code(x.dtype), batch, length, row_stride, k,
                    _order_code(sorted_index), int(bool(return_value)),
                    INDEX_INT64 if index_dtype == torch.int64 else INDEX_INT32,
                    vals.data_ptr() if (return_value and vals is not None) else None,
                    idx.data_ptr(), flag.data_ptr(), s.cuda_stream)
    if rc != OK:
        raise DsTopkError(rc)
    return vals, idx


def sample(x: torch.Tensor, k: int, temperature: float, top_p: float, u: torch.Tensor,
           nan_flag: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Sampler tail on a CUDA tensor x [batch, len] (contiguous rows): TopK in value order, temperature softmax over the k survivors, top-p
    nucleus, one draw per row with the caller's uniform numbers u (float32 CUDA
    [batch], each in [0, 1)). Returns (tokens int32 [batch], values [batch, k],
    indices int32 [batch, k])."""
    if x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a 2-D CUDA tensor with contiguous rows")
    if u.dtype != torch.float32 or not u.is_cuda or u.numel() != x.shape[0]:
        raise ValueError("u must be a float32 CUDA tensor with one number per row")
    batch, length = x.shape
    row_stride = x.stride(0) if batch > 1 else -(-length * x.element_size() // 16) * 16 // x.element_size()
    vals = torch.empty((batch, k), dtype=x.dtype, device=x.device)
    idx = torch.empty((batch, k), dtype=torch.int32, device=x.device)
    tokens = torch.empty(batch, dtype=torch.int32, device=x.device)
    flag = nan_flag if nan_flag is not None else torch.zeros(1, dtype=torch.int32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    rc = ds_topk_sample(x.data_ptr(), dtype_code(x.dtype), batch, length, row_stride, k,
                        float(temperature), float(top_p), u.contiguous().data_ptr(), vals.data_ptr(),
                        idx.data_ptr(), tokens.data_ptr(), flag.data_ptr(), s.cuda_stream)
    if rc != OK:
        raise DsTopkError(rc)
    return tokens, vals, idx
