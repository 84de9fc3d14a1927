"""CPU oracle for DeepSelect top-k -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never
calls it, and it never calls the product library: the two share no code.

The arithmetic lives in ``ds_oracle.c`` (plain single-threaded C); this module
only compiles it with gcc and marshals numpy arrays through ctypes.

What each function follows (page title, section):
  * ``topk``        -- the plain definition of top-k, milkfeng.top
                       "CUDA 算子笔记 4", section "Top K Selection", with ties
                       broken by lower index.
  * ``model``       -- the scan / filter / compact loop and its counters
                       A, R, W, peak; PFCCLab/DeepSelect "DeepSelect-deep-dive",
                       sections "算法" and "RadixSelectTopK 总处理元素数的期望上界".
  * ``keys``        -- the order-preserving float -> unsigned key map,
                       "CUDA 算子笔记 4", sub-section "改造 Radix Sort".
  * ``philox``      -- Philox4x32-10 (Salmon et al., SC'11).
  * ``permutation`` -- the input-independent block order built from it.

All of them are pinned by the ``-m "not gpu"`` tests (worked example, brute
force, closed forms, library routines); none is "parity unpinned".
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libds_oracle.so")

FP32 = 0
BF16 = 1
FP16 = 2
_DTYPE_CODES = {"fp32": FP32, "bf16": BF16, "fp16": FP16, FP32: FP32, BF16: BF16, FP16: FP16}

_lock = threading.Lock()
_lib = None


def build(force=False, src=_SRC, out=_LIB_PATH):
    """Compile the oracle with gcc (plain C, -O2, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src],
                   check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    c_i32p = ctypes.POINTER(ctypes.c_int32)
    c_u32p = ctypes.POINTER(ctypes.c_uint32)
    c_i64p = ctypes.POINTER(ctypes.c_int64)
    lib.ds_oracle_key_f32.argtypes = [ctypes.c_uint32]
    lib.ds_oracle_key_f32.restype = ctypes.c_uint32
    lib.ds_oracle_key_bf16.argtypes = [ctypes.c_uint32]
    lib.ds_oracle_key_bf16.restype = ctypes.c_uint32
    lib.ds_oracle_key_f16.argtypes = [ctypes.c_uint32]
    lib.ds_oracle_key_f16.restype = ctypes.c_uint32
    lib.ds_oracle_keys.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, c_u32p]
    lib.ds_oracle_keys.restype = None
    lib.ds_oracle_topk.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, c_i32p,
                                   ctypes.c_int64, ctypes.c_int, c_i32p, ctypes.c_void_p]
    lib.ds_oracle_topk.restype = ctypes.c_int
    lib.ds_oracle_philox4x32_10.argtypes = [c_u32p, c_u32p, c_u32p]
    lib.ds_oracle_philox4x32_10.restype = None
    lib.ds_oracle_permutation.argtypes = [ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint32,
                                          ctypes.c_uint32, ctypes.c_uint32, c_u32p]
    lib.ds_oracle_permutation.restype = ctypes.c_int
    lib.ds_oracle_model.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, c_i32p,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_uint64, ctypes.c_int, ctypes.c_int, c_i32p,
                                    ctypes.c_void_p, c_i64p]
    lib.ds_oracle_model.restype = ctypes.c_int
    lib.ds_oracle_sweep_f32.argtypes = []
    lib.ds_oracle_sweep_f32.restype = ctypes.c_int64
    return lib


def load(path=None):
    """Build if needed and load the oracle library (cached)."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_bits(x, dtype):
    """x as a C-contiguous array of raw bit patterns (uint32 for fp32, uint16 for bf16 / fp16)."""
    code = _DTYPE_CODES[dtype]
    want = np.uint32 if code == FP32 else np.uint16
    a = np.asarray(x)
    if a.dtype == np.float32 and code == FP32:
        a = a.view(np.uint32)
    if a.dtype == np.float16 and code == FP16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError("expected %s bit patterns, got %s" % (want, a.dtype))
    return np.ascontiguousarray(a), code


def _row_len(row_len, rows):
    if row_len is None:
        return None
    rl = np.ascontiguousarray(np.asarray(row_len, dtype=np.int32))
    if rl.shape != (rows,):
        raise ValueError("row_len must have one entry per row")
    return rl


def topk(x, dtype, k, row_len=None, lib=None):
    """Exact top-k of every row of a [rows, N] array of bit patterns.

    Returns (idx int32 [rows, k], val bits [rows, k]) sorted by value
    descending, ties by lower index; rows shorter than k are padded with
    index -1 and -inf.
    """
    lib = lib or load()
    bits, code = _as_bits(x, dtype)
    rows, N = bits.shape
    rl = _row_len(row_len, rows)
    out_idx = np.empty((rows, k), dtype=np.int32)
    out_val = np.empty((rows, k), dtype=bits.dtype)
    rc = lib.ds_oracle_topk(bits.ctypes.data, code, rows,
                            None if rl is None else _ptr(rl, ctypes.c_int32), N, k,
                            _ptr(out_idx, ctypes.c_int32), out_val.ctypes.data)
    if rc != 0:
        raise ValueError("ds_oracle_topk rejected its arguments")
    return out_idx, out_val


def model(x, dtype, k, B, B2, seed, row_len=None, splits=1, identity_order=False, lib=None):
    """Run the DeepSelect loop step by step.

    Returns (idx, val, stats) where stats is int64 [rows, splits, 4] holding
    (A, R, W, peak) of every slice.
    """
    lib = lib or load()
    bits, code = _as_bits(x, dtype)
    rows, N = bits.shape
    rl = _row_len(row_len, rows)
    out_idx = np.empty((rows, k), dtype=np.int32)
    out_val = np.empty((rows, k), dtype=bits.dtype)
    stats = np.zeros((rows, splits, 4), dtype=np.int64)
    rc = lib.ds_oracle_model(bits.ctypes.data, code, rows,
                             None if rl is None else _ptr(rl, ctypes.c_int32), N, k, B, B2,
                             ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), splits,
                             1 if identity_order else 0, _ptr(out_idx, ctypes.c_int32),
                             out_val.ctypes.data, _ptr(stats, ctypes.c_int64))
    if rc != 0:
        raise ValueError("ds_oracle_model rejected its arguments")
    return out_idx, out_val, stats


def keys(x, dtype, lib=None):
    """Order-preserving unsigned keys of an array of bit patterns."""
    lib = lib or load()
    bits, code = _as_bits(np.ravel(x), dtype)
    out = np.empty(bits.shape, dtype=np.uint32)
    lib.ds_oracle_keys(bits.ctypes.data, code, bits.size, _ptr(out, ctypes.c_uint32))
    return out.reshape(np.shape(x))


def philox(ctr, key, lib=None):
    """Philox4x32-10 of one 4-word counter under one 2-word key."""
    lib = lib or load()
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    kk = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.empty(4, dtype=np.uint32)
    lib.ds_oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(kk, ctypes.c_uint32),
                                _ptr(out, ctypes.c_uint32))
    return out


def permutation(m, seed, row=0, slice_=0, first_block=0, lib=None):
    """Visit order of blocks first_block .. first_block+m-1 of (row, slice)."""
    lib = lib or load()
    out = np.empty(max(m, 1), dtype=np.uint32)
    rc = lib.ds_oracle_permutation(m, ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), row,
                                   slice_, first_block, _ptr(out, ctypes.c_uint32))
    if rc != 0:
        raise MemoryError("ds_oracle_permutation failed")
    return out[:m]
