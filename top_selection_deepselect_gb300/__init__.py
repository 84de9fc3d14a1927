"""DeepSelect top-k for GB300 (sm_103a).

The product is the C-ABI library libds_topk.so (include/ds_topk.h), built
from hand-written CUDA in csrc/.  This package is its thin Python binding:
the functions named like the C entry points marshal arguments and raise on a
non-zero status; `topk` wraps them for torch tensors.  There is no CPU
fallback: without the compiled library every call raises.
"""
from ._binding import (DS_BF16, DS_ECUDA, DS_EINVAL, DS_EUNSUPPORTED, DS_FP16, DS_FP32, DS_OK,
                       DS_ORDER_IDENTITY, DS_ORDER_RANDOM, ENTRY_POINTS, DSError,
                       ds_last_error_detail, ds_strerror, ds_topk, ds_topk_ex, ds_topk_host,
                       ds_topk_host_async, ds_topk_long_row, ds_topk_long_row_noalloc,
                       ds_topk_long_row_workspace, ds_topk_max_k, ds_topk_plan,
                       ds_topk_stats_order, library_path, load_library, row_range, topk,
                       topk_long_row)
from ._build import build

__all__ = ["DS_BF16", "DS_ECUDA", "DS_EINVAL", "DS_EUNSUPPORTED", "DS_FP16", "DS_FP32", "DS_OK",
           "DS_ORDER_IDENTITY", "DS_ORDER_RANDOM", "ENTRY_POINTS", "DSError", "build",
           "ds_last_error_detail", "ds_strerror", "ds_topk", "ds_topk_ex", "ds_topk_host",
           "ds_topk_host_async", "ds_topk_long_row", "ds_topk_long_row_noalloc",
           "ds_topk_long_row_workspace", "ds_topk_max_k", "ds_topk_plan", "ds_topk_stats_order",
           "library_path", "load_library", "row_range", "topk", "topk_long_row"]
