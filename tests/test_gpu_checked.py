"""Bounds-checked build on the GPU.

The library is rebuilt with -DDS_CHECKED: every computed shared-memory range
that a write could overrun (appends into the candidate buffer, the select's
tie gather and compaction, the split-row copies into CTA 0) is checked; a
failed check records a bit in a device word and skips the write.  The cases
below must give the oracle's answer with the word still zero.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 0x5EED5EED


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import top_selection_deepselect_gb300 as ds
    from top_selection_deepselect_gb300 import _build
    d = tmp_path_factory.mktemp("checked")
    objs, procs = [], []
    for src in _build.SOURCES:
        obj = str(d / (os.path.basename(src) + ".o"))
        objs.append(obj)
        procs.append(subprocess.Popen([_build.nvcc()] + _build.NVCC_FLAGS +
                                      ["-DDS_CHECKED", "-I", _build.INCLUDE, "-c", "-o", obj, src]))
    assert all(p.wait() == 0 for p in procs)
    out = str(d / "libds_topk_checked.so")
    subprocess.run([_build.nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", out]
                   + objs, check=True)
    lib = ds.load_library(out)
    lib.ds_check_word.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.ds_check_word.restype = ctypes.c_int
    return lib


def check_word(lib):
    w = ctypes.c_uint32(0xFFFFFFFF)
    assert lib.ds_check_word(ctypes.addressof(w), 1) == 0
    return w.value


def run(lib, bits, dtype, k, B, B2, row_len=None, splits=0):
    rows, N = bits.shape
    if dtype == "fp32":
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).cuda()
    else:
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    code = {"fp32": 0, "bf16": 1, "fp16": 2}[dtype]
    rl = None if row_len is None else torch.from_numpy(np.asarray(row_len, np.int32)).cuda()
    oi = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ov = torch.empty((rows, k), dtype=x.dtype, device="cuda")
    rc = lib.ds_topk_ex(x.data_ptr(), code, rows, None if rl is None else rl.data_ptr(), N, k, B, B2,
                        ctypes.c_uint64(SEED), splits, oi.data_ptr(), ov.data_ptr(), None, None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return oi.cpu().numpy(), ov.cpu().numpy().view(bits.dtype)


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
@pytest.mark.parametrize("splits", [0, 1])
def test_workloads_pass_the_bounds_checks(lib, name, splits):
    c = workloads.CONFIGS[name]
    bits, row_len = workloads.config_inputs(name, rows=min(8, workloads.CONFIGS[name]["rows"]))
    ref_idx, ref_val = oracle.topk(bits, c["dtype"], c["k"], row_len=row_len)
    check_word(lib)
    idx, val = run(lib, bits, c["dtype"], c["k"], c["B"], c["B2"], row_len=row_len, splits=splits)
    assert check_word(lib) == 0
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_array_equal(val, ref_val)


@pytest.mark.parametrize("kind", ["specials", "levels", "constant", "ascending"])
def test_edge_cases_pass_the_bounds_checks(lib, kind):
    bits, _ = workloads.generate(6, 30000, "bf16", kind, seed=53, fraction=0.2, value=2.0)
    row_len = np.array([30000, 0, 1, 700, 12345, 29999], dtype=np.int32)
    for k, B, B2, splits in [(1, 64, 64, 1), (64, 128, 128, 16), (777, 512, 128, 3),
                             (1100, 512, 512, 8), (900, 512, 512, 7), (3000, 1024, 1024, 2),
                             (5000, 1024, 1024, 1)]:
        ref_idx, ref_val = oracle.topk(bits, "bf16", k, row_len=row_len)
        check_word(lib)
        idx, val = run(lib, bits, "bf16", k, B, B2, row_len=row_len, splits=splits)
        assert check_word(lib) == 0, (k, B, B2, splits)
        np.testing.assert_array_equal(idx, ref_idx)
        np.testing.assert_array_equal(val, ref_val)


@pytest.mark.parametrize("dtype,N,k,B,B2", [("fp32", 3_000_017, 512, 1024, 1024),
                                            ("bf16", 1_048_577, 16, 8192, 1024)])
def test_long_row_passes_the_bounds_checks(lib, dtype, N, k, B, B2):
    # both launches of a long-row call, including a last piece shorter than P
    lib.ds_topk_long_row_workspace.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]
    lib.ds_topk_long_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p,
                                     ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p]
    code = {"fp32": 0, "bf16": 1}[dtype]
    bits, _ = workloads.generate(1, N, dtype, "normal", seed=54)
    x = torch.from_numpy(bits.reshape(-1).view(np.int32 if dtype == "fp32" else np.int16)).cuda()
    nb, G = ctypes.c_size_t(0), ctypes.c_int(0)
    assert lib.ds_topk_long_row_workspace(code, N, k, B, B2, ctypes.byref(nb), None,
                                          ctypes.byref(G)) == 0
    assert G.value > 1
    ws = torch.empty(nb.value, dtype=torch.uint8, device="cuda")
    oi = torch.empty(k, dtype=torch.int32, device="cuda")
    ov = torch.empty(k, dtype=x.dtype, device="cuda")
    check_word(lib)
    rc = lib.ds_topk_long_row(x.data_ptr(), code, N, k, B, B2, ctypes.c_uint64(SEED),
                              ws.data_ptr(), nb.value, oi.data_ptr(), ov.data_ptr(), None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert check_word(lib) == 0
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    np.testing.assert_array_equal(oi.cpu().numpy(), ref_idx[0])
    np.testing.assert_array_equal(ov.cpu().numpy().view(bits.dtype), ref_val[0])
