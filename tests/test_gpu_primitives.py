"""Device primitives against the pages' worked examples (GPU).

The scan and compaction examples of elainafan.one "并行算法（一）" (sections
"Scan" and "Compact") are stored in tests/golden/; a small test library built
from tests/primitives_kernels.cu runs the library's own warp scan, its
ballot-rank compaction and its __ffs mask walk on them.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def golden(name):
    fields = {}
    for line in open(os.path.join(HERE, "golden", name)):
        if line.startswith("#") or ":" not in line:
            continue
        key, val = line.split(":", 1)
        fields[key.strip()] = [int(v) for v in val.split()]
    return fields


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from top_selection_deepselect_gb300 import _build
    out = str(tmp_path_factory.mktemp("prim") / "libprim.so")
    subprocess.run([_build.nvcc()] + _build.NVCC_FLAGS +
                   ["-shared", "-I", os.path.join(ROOT, "top_selection_deepselect_gb300", "csrc"),
                    "-o", out, os.path.join(HERE, "primitives_kernels.cu")], check=True)
    lib = ctypes.CDLL(out)
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32
    lib.prim_scan.argtypes = [vp, i32, vp, vp]
    lib.prim_compact.argtypes = [vp, vp, i32, vp, vp]
    lib.prim_mask_walk.argtypes = [vp, u32, vp, vp]
    lib.prim_block_order.argtypes = [u32, u32, vp]
    return lib


def dev(a, dtype=torch.int32):
    return torch.tensor(a, dtype=dtype, device="cuda")


def test_warp_scan_matches_the_pages_example(lib):
    g = golden("scan_example.txt")
    x = dev(g["input"])
    incl = torch.zeros_like(x)
    excl = torch.zeros_like(x)
    assert lib.prim_scan(x.data_ptr(), len(g["input"]), incl.data_ptr(), excl.data_ptr()) == 0
    assert incl.cpu().tolist() == g["inclusive"]
    assert excl.cpu().tolist() == g["exclusive"]


def test_ballot_compaction_matches_the_pages_example(lib):
    g = golden("compact_example.txt")
    x, p = dev(g["x"]), dev(g["p"])
    out = torch.zeros(32, dtype=torch.int64, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.prim_compact(x.data_ptr(), p.data_ptr(), len(g["x"]), out.data_ptr(), count.data_ptr()) == 0
    n = int(count.item())
    assert n == sum(g["p"]) == len(g["output"])
    assert out[:n].cpu().tolist() == g["output"]
    # the slots are the exclusive scan of the flags
    assert np.cumsum([0] + g["p"][:-1]).tolist() == g["scan"]


def test_ffs_mask_walk_matches_the_pages_example(lib):
    g = golden("compact_example.txt")
    x = dev(g["x"])
    mask = sum(1 << i for i, f in enumerate(g["p"]) if f)
    out = torch.zeros(32, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.prim_mask_walk(x.data_ptr(), mask, out.data_ptr(), count.data_ptr()) == 0
    n = int(count.item())
    assert out[:n].cpu().tolist() == g["output"]


def test_block_order_is_a_permutation(lib):
    """The free-running kernel's block order (keyed Feistel network, cycle
    walked) maps the positions 0..n-1 onto the block ids 0..n-1 exactly once,
    for sizes around powers of four (the network's domains) and several keys."""
    for n in [1, 2, 3, 4, 5, 15, 16, 17, 31, 63, 64, 65, 125, 255, 256, 257, 1000, 1024, 1025,
              4095, 4096, 65537]:
        for word in [0, 1, 0x5EED5EED, 0xFFFFFFFF]:
            out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
            assert lib.prim_block_order(n, word, out.data_ptr()) == 0
            got = np.sort(out.cpu().numpy())
            np.testing.assert_array_equal(got, np.arange(n, dtype=np.int32))


def test_block_order_spreads_positions(lib):
    """Where block 0 lands over many keys: its mean position is near the middle
    (the order depends on the key, not on the data), and the keys give
    different orders."""
    n = 125
    pos0, firsts = [], set()
    for word in range(400):
        out = torch.empty(n, dtype=torch.int32, device="cuda")
        assert lib.prim_block_order(n, word * 2654435761 % (1 << 32), out.data_ptr()) == 0
        o = out.cpu().numpy()
        pos0.append(int(np.nonzero(o == 0)[0][0]))
        firsts.add(int(o[0]))
    assert abs(np.mean(pos0) - (n - 1) / 2) < 8  # 400 draws: standard error about 1.8
    assert len(firsts) > 60
