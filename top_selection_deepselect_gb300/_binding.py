"""ctypes binding of libds_topk.so -- argument marshalling only.

Every function named like a C entry point of include/ds_topk.h takes the same
arguments (device pointers as Python ints, the stream as a cudaStream_t
handle) and raises DSError on a non-zero status.  `topk` is a convenience
wrapper that takes torch tensors, allocates the outputs with torch and calls
ds_topk_ex on the tensor's current stream.  All computation happens in the
CUDA library; if it cannot be loaded, every call raises.
"""
import ctypes
import os
import threading

from . import _build

DS_OK = 0
DS_EINVAL = -1
DS_EUNSUPPORTED = -2
DS_ECUDA = -3
DS_FP32 = 0
DS_BF16 = 1
DS_FP16 = 2
DS_ORDER_RANDOM = 0
DS_ORDER_IDENTITY = 1

ENTRY_POINTS = ["ds_topk", "ds_topk_ex", "ds_topk_stats_order", "ds_topk_host", "ds_topk_host_async", "ds_topk_long_row",
                "ds_topk_long_row_workspace", "ds_topk_long_row_noalloc", "ds_topk_plan",
                "ds_topk_max_k", "ds_strerror", "ds_last_error_detail"]


class DSError(RuntimeError):
    """A non-zero status from libds_topk."""

    def __init__(self, status, where, detail):
        self.status = status
        super().__init__("%s failed: %s (%d)%s" % (where, _strerror_safe(status), status,
                                                   (": " + detail) if detail else ""))


class ds_plan_t(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in
                ("splits", "threads", "stages", "blocks_per_stage", "warps_per_block", "async_copy",
                 "smem_bytes", "capacity", "grid", "ctas_per_sm", "kernel")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def library_path():
    return _build.LIB_PATH


def load_library(path=None):
    """Load libds_topk.so (built by __graft_entry__.build()); raises if missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libds_topk.so is not built (%s); run __graft_entry__.build()" % p)
        lib = ctypes.CDLL(p)
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        lib.ds_topk.argtypes = [vp, i32, i32, vp, i64, i32, i32, i32, u64, vp, vp, vp]
        lib.ds_topk.restype = i32
        lib.ds_topk_ex.argtypes = [vp, i32, i32, vp, i64, i32, i32, i32, u64, i32, vp, vp, vp, vp]
        lib.ds_topk_ex.restype = i32
        lib.ds_topk_stats_order.argtypes = [vp, i32, i32, vp, i64, i32, i32, i32, u64, i32, i32,
                                            vp, vp, vp, vp]
        lib.ds_topk_stats_order.restype = i32
        lib.ds_topk_host.argtypes = [vp, i32, i32, vp, i64, i32, i32, i32, u64, vp, vp,
                                     vp, vp, vp, vp, vp]
        lib.ds_topk_host.restype = i32
        lib.ds_topk_host_async.argtypes = [vp, i32, i32, vp, i64, i32, i32, i32, u64, vp, vp,
                                           vp, vp, vp, vp, vp]
        lib.ds_topk_host_async.restype = i32
        lib.ds_topk_long_row.argtypes = [vp, i32, i64, i32, i32, i32, u64, vp, ctypes.c_size_t,
                                         vp, vp, vp]
        lib.ds_topk_long_row.restype = i32
        lib.ds_topk_long_row_workspace.argtypes = [i32, i64, i32, i32, i32,
                                                   ctypes.POINTER(ctypes.c_size_t),
                                                   ctypes.POINTER(ctypes.c_int64),
                                                   ctypes.POINTER(ctypes.c_int)]
        lib.ds_topk_long_row_workspace.restype = i32
        lib.ds_topk_long_row_noalloc.argtypes = [vp, i32, i64, i32, i32, i32, u64, vp, vp, vp]
        lib.ds_topk_long_row_noalloc.restype = i32
        lib.ds_topk_plan.argtypes = [vp, i32, i32, i64, i32, i32, i32, i32,
                                     ctypes.POINTER(ds_plan_t)]
        lib.ds_topk_plan.restype = i32
        lib.ds_topk_max_k.argtypes = [i32, i32, i32]
        lib.ds_topk_max_k.restype = i32
        lib.ds_strerror.argtypes = [i32]
        lib.ds_strerror.restype = ctypes.c_char_p
        lib.ds_last_error_detail.argtypes = []
        lib.ds_last_error_detail.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _strerror_safe(status):
    try:
        return load_library().ds_strerror(status).decode()
    except Exception:
        return "status"


def _check(status, where):
    if status != DS_OK:
        detail = load_library().ds_last_error_detail().decode()
        raise DSError(status, where, detail)
    return status


def _u64(seed):
    return ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF)


# ---- C entry points, same names and argument order ---------------------------
def ds_topk(x, dtype, rows, row_len, N, k, B, B2, seed, out_idx, out_val, stream):
    return _check(load_library().ds_topk(x, dtype, rows, row_len, N, k, B, B2, _u64(seed),
                                          out_idx, out_val, stream), "ds_topk")


def ds_topk_ex(x, dtype, rows, row_len, N, k, B, B2, seed, splits, out_idx, out_val, stats,
               stream):
    return _check(load_library().ds_topk_ex(x, dtype, rows, row_len, N, k, B, B2, _u64(seed),
                                             splits, out_idx, out_val, stats, stream),
                  "ds_topk_ex")


def ds_topk_stats_order(x, dtype, rows, row_len, N, k, B, B2, seed, splits, order, out_idx,
                        out_val, stats, stream):
    return _check(load_library().ds_topk_stats_order(x, dtype, rows, row_len, N, k, B, B2,
                                                      _u64(seed), splits, order, out_idx, out_val,
                                                      stats, stream),
                  "ds_topk_stats_order")


def row_range(rank, world, rows):
    """Contiguous rows [r0, r1) of `rows` that rank `rank` of `world` selects
    when a batch is split across GPUs: rows are independent, so every rank
    calls ds_topk on its own slice and writes its own slice of the outputs;
    the first rows % world ranks take one row more."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("need 0 <= rank < world and rows >= 0")
    base, extra = divmod(rows, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def ds_topk_host(x_host, dtype, rows, row_len_host, N, k, B, B2, seed, out_idx_host,
                 out_val_host, x_dev, row_len_dev, out_idx_dev, out_val_dev, stream):
    return _check(load_library().ds_topk_host(x_host, dtype, rows, row_len_host, N, k, B, B2,
                                               _u64(seed), out_idx_host, out_val_host, x_dev,
                                               row_len_dev, out_idx_dev, out_val_dev, stream),
                  "ds_topk_host")


def ds_topk_host_async(x_host, dtype, rows, row_len_host, N, k, B, B2, seed, out_idx_host,
                       out_val_host, x_dev, row_len_dev, out_idx_dev, out_val_dev, stream):
    return _check(load_library().ds_topk_host_async(x_host, dtype, rows, row_len_host, N, k, B, B2,
                                                     _u64(seed), out_idx_host, out_val_host, x_dev,
                                                     row_len_dev, out_idx_dev, out_val_dev, stream),
                  "ds_topk_host_async")


def ds_topk_long_row(x, dtype, N, k, B, B2, seed, workspace, workspace_bytes, out_idx, out_val,
                     stream):
    return _check(load_library().ds_topk_long_row(x, dtype, N, k, B, B2, _u64(seed), workspace,
                                                   workspace_bytes, out_idx, out_val, stream),
                  "ds_topk_long_row")


def ds_topk_long_row_workspace(dtype, N, k, B, B2, plan=False):
    """Workspace bytes; with plan=True, (bytes, piece length P, pieces G)."""
    n, P, G = ctypes.c_size_t(0), ctypes.c_int64(0), ctypes.c_int(0)
    _check(load_library().ds_topk_long_row_workspace(dtype, N, k, B, B2, ctypes.byref(n),
                                                     ctypes.byref(P), ctypes.byref(G)),
           "ds_topk_long_row_workspace")
    return (n.value, P.value, G.value) if plan else n.value


def ds_topk_long_row_noalloc(x, dtype, N, k, B, B2, seed, out_idx, out_val, stream):
    return _check(load_library().ds_topk_long_row_noalloc(x, dtype, N, k, B, B2, _u64(seed),
                                                           out_idx, out_val, stream),
                  "ds_topk_long_row_noalloc")


def ds_topk_plan(x, dtype, rows, N, k, B, B2, splits=0):
    plan = ds_plan_t()
    _check(load_library().ds_topk_plan(x, dtype, rows, N, k, B, B2, splits, ctypes.byref(plan)),
           "ds_topk_plan")
    return plan.as_dict()


def ds_topk_max_k(dtype, B, B2):
    r = load_library().ds_topk_max_k(dtype, B, B2)
    if r < 0:
        _check(r, "ds_topk_max_k")
    return r


def ds_strerror(status):
    return load_library().ds_strerror(status).decode()


def ds_last_error_detail():
    return load_library().ds_last_error_detail().decode()


# ---- torch convenience wrapper ----------------------------------------------
def dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return DS_FP32
    if t.dtype == torch.bfloat16:
        return DS_BF16
    if t.dtype == torch.float16:
        return DS_FP16
    raise TypeError("x must be float32, bfloat16 or float16, got %s" % t.dtype)


def topk(x, k, B, B2, seed=0x5EED5EED, row_len=None, splits=0, stats=False, out_idx=None,
         out_val=None, stream=None, order=None):
    """Top-k of every row of a 2-D CUDA tensor x (float32, bfloat16 or float16).

    Returns (idx int32 [rows, k], val [rows, k]) and, with stats=True, also an
    int64 [rows, splits, 4] tensor of (A, R, W, peak) per slice.  `order`
    (DS_ORDER_RANDOM or DS_ORDER_IDENTITY, with stats=True) calls
    ds_topk_stats_order.
    """
    import torch
    if x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2-D CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous (row pitch = N)")
    rows, N = x.shape
    code = dtype_code(x)
    if out_idx is None:
        out_idx = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    if out_val is None:
        out_val = torch.empty((rows, k), dtype=x.dtype, device=x.device)
    rl_ptr = None
    if row_len is not None:
        if row_len.dtype != torch.int32 or not row_len.is_cuda or row_len.numel() != rows:
            raise ValueError("row_len must be a CUDA int32 tensor with one entry per row")
        rl_ptr = row_len.data_ptr()
    st_t = None
    if stats:
        if splits < 1:
            raise ValueError("stats need an explicit splits >= 1")
        st_t = torch.zeros((rows, splits, 4), dtype=torch.int64, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    if order is not None:
        if not stats:
            raise ValueError("order needs stats=True")
        ds_topk_stats_order(x.data_ptr(), code, rows, rl_ptr, N, k, B, B2, seed, splits, order,
                            out_idx.data_ptr(), out_val.data_ptr(), st_t.data_ptr(),
                            stream.cuda_stream)
    else:
        ds_topk_ex(x.data_ptr(), code, rows, rl_ptr, N, k, B, B2, seed, splits,
                   out_idx.data_ptr(), out_val.data_ptr(),
                   None if st_t is None else st_t.data_ptr(), stream.cuda_stream)
    if stats:
        return out_idx, out_val, st_t
    return out_idx, out_val


def topk_long_row(x, k, B, B2, seed=0x5EED5EED, workspace=None, out_idx=None, out_val=None,
                  stream=None):
    """Top-k of one long 1-D CUDA tensor x spread over the whole GPU.

    Returns (idx int32 [k], val [k]).  The workspace (a CUDA uint8 tensor of
    at least ds_topk_long_row_workspace bytes) is allocated with torch when not
    given.
    """
    import torch
    if x.dim() != 1 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous 1-D CUDA tensor")
    N = x.numel()
    code = dtype_code(x)
    need = ds_topk_long_row_workspace(code, N, k, B, B2)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    elif workspace.numel() < need:
        raise ValueError("workspace has %d bytes, %d needed" % (workspace.numel(), need))
    if out_idx is None:
        out_idx = torch.empty(k, dtype=torch.int32, device=x.device)
    if out_val is None:
        out_val = torch.empty(k, dtype=x.dtype, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    ds_topk_long_row(x.data_ptr(), code, N, k, B, B2, seed, workspace.data_ptr(),
                     workspace.numel(), out_idx.data_ptr(), out_val.data_ptr(), stream.cuda_stream)
    return out_idx, out_val
