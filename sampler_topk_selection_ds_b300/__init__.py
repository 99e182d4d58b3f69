"""B300-native batched row-wise TopK (bf16 Lightning-Indexer scores, fp32 sampler logits).

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
libds_topk.so (include/ds_topk.h); this package is its thin ctypes binding.
"""
from ._binding import (BF16, EALIGN, ECUDA, EINVAL, ETIMEOUT, FLAG_NAN, FLAG_TIMEOUT, FP32,
                       INDEX_INT32, INDEX_INT64, LIB_PATH, MAX_K, OK, PATH_CLUSTER, PATH_ROW, PATH_WARP_ROWS, SORT_INDEX, SORT_NONE, SORT_VALUE,
                       DsTopkError, Plan, ds_topk,
                       ds_topk_ex, ds_topk_plan, ds_topk_sample, dtype_code, sample, status_string, topk, version)

__all__ = ["BF16", "FP32", "OK", "EINVAL", "EALIGN", "ECUDA", "ETIMEOUT", "FLAG_NAN",
           "FLAG_TIMEOUT", "INDEX_INT32", "INDEX_INT64", "MAX_K", "PATH_ROW", "PATH_CLUSTER", "PATH_WARP_ROWS", "SORT_NONE", "SORT_INDEX", "SORT_VALUE", "LIB_PATH", "DsTopkError", "Plan",
           "ds_topk", "ds_topk_ex", "ds_topk_plan", "ds_topk_sample", "dtype_code", "sample", "status_string", "topk",
           "version"]
