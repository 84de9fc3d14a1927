"""The C-ABI library builds, loads and exports what include/ds_topk.h declares;
argument checks answer before any CUDA call (CPU only, no compute)."""
import ctypes
import os
import re

import pytest

import top_selection_deepselect_gb300 as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds_topk.h")


@pytest.fixture(scope="module")
def lib():
    ds.build()
    return ds.load_library()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ds_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert names == sorted(ds.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_is_built_for_sm_103a(lib):
    # nvcc flags used by the build: one -gencode for compute_103a / sm_103a
    from top_selection_deepselect_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in _build.NVCC_FLAGS
    assert "--use_fast_math" not in _build.NVCC_FLAGS


def test_dtype_codes():
    # fp32, bf16 and IEEE fp16 are the dtypes of include/ds_topk.h
    assert (ds.DS_FP32, ds.DS_BF16, ds.DS_FP16) == (0, 1, 2)
    with open(HEADER) as f:
        text = f.read()
    assert "#define DS_FP16 2" in text


def test_strerror_texts(lib):
    for status in [ds.DS_OK, ds.DS_EINVAL, ds.DS_EUNSUPPORTED, ds.DS_ECUDA]:
        assert ds.ds_strerror(status)
    assert ds.ds_strerror(-99) == "unknown status"


FAKE = 1 << 20  # never dereferenced: these calls fail their checks first


@pytest.mark.parametrize("args,status", [
    (dict(dtype=7), ds.DS_EUNSUPPORTED),
    (dict(dtype=3), ds.DS_EUNSUPPORTED),
    (dict(rows=-1), ds.DS_EINVAL),
    (dict(N=0), ds.DS_EINVAL),
    (dict(N=1 << 31), ds.DS_EINVAL),
    (dict(k=0), ds.DS_EINVAL),
    (dict(k=1025, N=1024), ds.DS_EINVAL),
    (dict(B=0), ds.DS_EINVAL),
    (dict(B2=0), ds.DS_EINVAL),
    (dict(splits=17), ds.DS_EINVAL),
    (dict(splits=-1), ds.DS_EINVAL),
    (dict(x=None), ds.DS_EINVAL),
    (dict(out_idx=None), ds.DS_EINVAL),
    (dict(out_val=None), ds.DS_EINVAL),
    (dict(stats=FAKE, splits=0), ds.DS_EINVAL),
])
def test_argument_errors_are_reported_before_any_launch(lib, args, status):
    a = dict(x=FAKE, dtype=ds.DS_FP32, rows=4, row_len=None, N=1024, k=8, B=128, B2=128,
             seed=1, splits=0, out_idx=FAKE, out_val=FAKE, stats=None, stream=None)
    a.update(args)
    rc = lib.ds_topk_ex(a["x"], a["dtype"], a["rows"], a["row_len"], a["N"], a["k"], a["B"],
                        a["B2"], ctypes.c_uint64(a["seed"]), a["splits"], a["out_idx"],
                        a["out_val"], a["stats"], a["stream"])
    assert rc == status
    assert ds.ds_last_error_detail()


@pytest.mark.parametrize("order,stats,splits", [(2, FAKE, 1), (-1, FAKE, 1), (0, None, 1),
                                                (1, None, 1), (1, FAKE, 0)])
def test_block_order_entry_checks_its_arguments(lib, order, stats, splits):
    """ds_topk_stats_order: a known order, counters (the order changes only
    them) and an explicit split factor, all refused before any launch."""
    rc = lib.ds_topk_stats_order(FAKE, ds.DS_FP32, 4, None, 1024, 8, 128, 128, ctypes.c_uint64(1),
                                 splits, order, FAKE, FAKE, stats, None)
    assert rc == ds.DS_EINVAL
    assert ds.ds_last_error_detail()


def test_zero_rows_is_a_noop(lib):
    assert lib.ds_topk(None, ds.DS_BF16, 0, None, 100, 5, 16, 16, ctypes.c_uint64(0),
                       None, None, None) == ds.DS_OK


def test_host_entry_checks_staging_buffers(lib):
    rc = lib.ds_topk_host(FAKE, ds.DS_FP32, 2, FAKE, 64, 4, 16, 16, ctypes.c_uint64(0),
                          FAKE, FAKE, FAKE, None, FAKE, FAKE, None)
    assert rc == ds.DS_EINVAL          # row_len_host given without row_len_dev
    rc = lib.ds_topk_host(FAKE, ds.DS_FP32, 2, None, 64, 4, 16, 16, ctypes.c_uint64(0),
                          FAKE, FAKE, None, None, FAKE, FAKE, None)
    assert rc == ds.DS_EINVAL          # no device staging for x
    for fn in (lib.ds_topk_host, lib.ds_topk_host_async):
        rc = fn(FAKE, ds.DS_FP32, 2, FAKE, 64, 4, 16, 16, ctypes.c_uint64(0),
                FAKE, FAKE, FAKE, None, FAKE, FAKE, None)
        assert rc == ds.DS_EINVAL      # row_len_host given without row_len_dev
        rc = fn(FAKE, ds.DS_FP32, 2, None, 64, 65, 16, 16, ctypes.c_uint64(0),
                FAKE, FAKE, FAKE, None, FAKE, FAKE, None)
        assert rc == ds.DS_EINVAL      # k > N


def test_python_wrapper_raises_with_detail(lib):
    with pytest.raises(ds.DSError) as e:
        ds.ds_topk_ex(FAKE, ds.DS_FP32, 1, None, 10, 11, 4, 4, 0, 0, FAKE, FAKE, None, None)
    assert e.value.status == ds.DS_EINVAL
    assert "k = 11" in str(e.value)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        ds.load_library(str(tmp_path / "absent.so"))


def test_no_cuda_device_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = lib.ds_topk(FAKE, ds.DS_FP32, 1, None, 1024, 8, 128, 128, ctypes.c_uint64(0), FAKE,
                     FAKE, None)
    assert rc == ds.DS_ECUDA


@pytest.mark.parametrize("args,status", [
    (dict(dtype=3), ds.DS_EUNSUPPORTED),
    (dict(N=0), ds.DS_EINVAL),
    (dict(N=1 << 31), ds.DS_EINVAL),
    (dict(k=0), ds.DS_EINVAL),
    (dict(k=2049, N=2048), ds.DS_EINVAL),
    (dict(B=0), ds.DS_EINVAL),
    (dict(B2=0), ds.DS_EINVAL),
    (dict(x=None), ds.DS_EINVAL),
    (dict(out_idx=None), ds.DS_EINVAL),
    (dict(out_val=None), ds.DS_EINVAL),
])
def test_long_row_argument_errors(lib, args, status):
    a = dict(x=FAKE, dtype=ds.DS_FP32, N=1 << 24, k=64, B=1024, B2=1024, out_idx=FAKE,
             out_val=FAKE)
    a.update(args)
    rc = lib.ds_topk_long_row(a["x"], a["dtype"], a["N"], a["k"], a["B"], a["B2"],
                              ctypes.c_uint64(0), FAKE, 1 << 20, a["out_idx"], a["out_val"], None)
    assert rc == status
    assert ds.ds_last_error_detail()
    rc = lib.ds_topk_long_row_noalloc(a["x"], a["dtype"], a["N"], a["k"], a["B"], a["B2"],
                                      ctypes.c_uint64(0), a["out_idx"], a["out_val"], None)
    assert rc == status
    if a["x"] and a["out_idx"] and a["out_val"]:
        # the workspace query makes the same argument checks (it has no pointers)
        n = ctypes.c_size_t(0)
        rc = lib.ds_topk_long_row_workspace(a["dtype"], a["N"], a["k"], a["B"], a["B2"],
                                            ctypes.byref(n), None, None)
        assert rc == status


def test_long_row_workspace_query_needs_an_output(lib):
    assert lib.ds_topk_long_row_workspace(ds.DS_FP32, 1 << 24, 64, 1024, 1024, None, None,
                                          None) == ds.DS_EINVAL
