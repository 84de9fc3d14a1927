"""GPU check of ds_topk_long_row_noalloc, the entry point that keeps the
long-row workspace in an array built into the library.  Its results must
equal those of ds_topk_long_row (caller-owned workspace) exactly -- the
result is unique -- on consecutive calls that reuse the built-in array.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SEED = 0x5EED5EED


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import top_selection_deepselect_gb300 as _ds
    _ds.build()
    _ds.load_library()
    return _ds


def device_input(N, dtype, kind, seed):
    bits, _ = workloads.generate(1, N, dtype, kind, seed=seed)
    if dtype == "fp32":
        return torch.from_numpy(bits.reshape(-1).view(np.int32)).to(DEV).view(torch.float32)
    return torch.from_numpy(bits.reshape(-1).view(np.int16)).to(DEV).view(torch.bfloat16)


def with_workspace(ds, x, code, k, B, B2):
    N = x.numel()
    nb = ds.ds_topk_long_row_workspace(code, N, k, B, B2)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    oi = torch.empty(k, dtype=torch.int32, device=DEV)
    ov = torch.empty(k, dtype=x.dtype, device=DEV)
    ds.ds_topk_long_row(x.data_ptr(), code, N, k, B, B2, SEED, ws.data_ptr(), nb, oi.data_ptr(),
                        ov.data_ptr(), None)
    torch.cuda.synchronize()
    return oi, ov


def test_no_alloc_entry_point_matches_the_workspace_entry_point(ds):
    lib = ds.load_library()
    cases = [(3_000_017, "fp32", "normal", 512, 1024, 1024, 71),
             (4_194_304, "bf16", "levels", 100, 1024, 1024, 72),
             (3_000_017, "fp32", "normal", 64, 1024, 1024, 73)]
    for N, dtype, kind, k, B, B2, seed in cases:      # consecutive calls share the array
        x = device_input(N, dtype, kind, seed)
        code = 0 if dtype == "fp32" else 1
        nb, P, G = ds.ds_topk_long_row_workspace(code, N, k, B, B2, plan=True)
        assert G > 1 and 0 < nb <= 8 << 20
        ref_i, ref_v = with_workspace(ds, x, code, k, B, B2)
        oi = torch.full((k,), -7, dtype=torch.int32, device=DEV)
        ov = torch.zeros(k, dtype=x.dtype, device=DEV)
        rc = lib.ds_topk_long_row_noalloc(x.data_ptr(), code, N, k, B, B2,
                                          ctypes.c_uint64(SEED), oi.data_ptr(), ov.data_ptr(),
                                          None)
        assert rc == 0, ds.ds_last_error_detail()
        torch.cuda.synchronize()
        assert torch.equal(oi, ref_i)
        assert torch.equal(ov.view(torch.int16 if dtype != "fp32" else torch.int32),
                           ref_v.view(torch.int16 if dtype != "fp32" else torch.int32))


def test_no_alloc_entry_point_on_a_row_selected_directly(ds):
    """A row shorter than 64 k is selected in one piece (G = 1): no workspace
    is needed, the built-in array is not used, and the result still equals
    the caller-workspace entry point's."""
    lib = ds.load_library()
    N, k = 5000, 100
    x = device_input(N, "fp32", "normal", 74)
    nb, P, G = ds.ds_topk_long_row_workspace(0, N, k, 1024, 1024, plan=True)
    assert G == 1 and nb == 0 and P == N
    ref_i, ref_v = with_workspace(ds, x, 0, k, 1024, 1024)
    for _ in range(2):
        oi = torch.full((k,), -7, dtype=torch.int32, device=DEV)
        ov = torch.zeros(k, dtype=torch.float32, device=DEV)
        rc = lib.ds_topk_long_row_noalloc(x.data_ptr(), 0, N, k, 1024, 1024, ctypes.c_uint64(SEED),
                                          oi.data_ptr(), ov.data_ptr(), None)
        assert rc == 0, ds.ds_last_error_detail()
        torch.cuda.synchronize()
        assert torch.equal(oi, ref_i)
        assert torch.equal(ov.view(torch.int32), ref_v.view(torch.int32))


def test_no_alloc_entry_point_refuses_more_than_its_workspace(ds):
    lib = ds.load_library()
    N, k = 1 << 26, 4096
    nb = ds.ds_topk_long_row_workspace(0, N, k, 1024, 1024)
    assert nb > 8 << 20
    x = torch.zeros(N, dtype=torch.float32, device=DEV)
    oi = torch.empty(k, dtype=torch.int32, device=DEV)
    ov = torch.empty(k, dtype=torch.float32, device=DEV)
    rc = lib.ds_topk_long_row_noalloc(x.data_ptr(), 0, N, k, 1024, 1024, ctypes.c_uint64(SEED),
                                      oi.data_ptr(), ov.data_ptr(), None)
    assert rc == ds.DS_EUNSUPPORTED
    assert "workspace" in ds.ds_last_error_detail()
