"""GPU parity of ds_topk_long_row (one row over the whole GPU) against the oracle.

The long-row path cuts the row into pieces, selects every piece, selects the
top k of the piece results and maps positions back to row indices.  Its
result is the row's unique top k, so indices and value bits must equal the
oracle's exactly, whatever the piece layout; the full-size case (the long-row
workload the benchmark times) is checked by properties that hold at any size.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ds = None


@pytest.fixture(scope="module", autouse=True)
def library():
    global ds
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import top_selection_deepselect_gb300 as _ds
    _ds.build()
    _ds.load_library()
    ds = _ds
    yield


DEV = "cuda:0"
SEED = 0x5EED5EED
CODE = {"fp32": 0, "bf16": 1, "fp16": 2}


def to_device(bits, dtype):
    if dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(DEV).view(torch.float32)
    t16 = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(t16)


def val_bits(t, dtype):
    if dtype == "fp32":
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def long_row(bits, dtype, k, B, B2, seed=SEED):
    x = to_device(bits.reshape(-1), dtype)
    idx, val = ds.topk_long_row(x, k, B, B2, seed=seed)
    torch.cuda.synchronize()
    return idx.cpu().numpy()[None, :], val_bits(val, dtype)[None, :]


def plan(dtype, N, k, B, B2):
    return ds.ds_topk_long_row_workspace(CODE[dtype], N, k, B, B2, plan=True)


def assert_same(idx, val, ref_idx, ref_val):
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_array_equal(val, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("N,k,B", [(3_000_017, 64, 1024), (1 << 22, 512, 1024),
                                   (5_000_011, 2048, 2048)])
def test_long_row_matches_the_oracle(dtype, N, k, B):
    _, P, G = plan(dtype, N, k, B, B)
    assert G > 1 and P % B == 0 and (G - 1) * P < N <= G * P
    bits, _ = workloads.generate(1, N, dtype, "normal", seed=61)
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    idx, val = long_row(bits, dtype, k, B, B)
    assert_same(idx, val, ref_idx, ref_val)


def test_last_piece_shorter_than_k():
    # pads of the short last piece tie with real -inf values and must lose.
    # Pieces are whole blocks, so large blocks and a small k leave a row of
    # (G-1) pieces plus one element for some lengths.
    k, B, B2 = 16, 8192, 1024
    for N in range((1 << 20) + 1, 8 << 20, B):
        nb, P, G = plan("fp32", N, k, B, B2)
        if G > 1 and N - (G - 1) * P < k:
            break
    else:
        pytest.fail("no length with a last piece shorter than k found")
    bits, _ = workloads.generate(1, N, "fp32", "normal", seed=62)
    ref_idx, ref_val = oracle.topk(bits, "fp32", k)
    assert_same(*long_row(bits, "fp32", k, B, B2), ref_idx, ref_val)
    # every element -inf: the answer is indices 0..k-1, never a pad
    ninf = np.full((1, N), 0xFF800000, dtype=np.uint32)
    idx, val = long_row(ninf, "fp32", k, B, B2)
    np.testing.assert_array_equal(idx[0], np.arange(k))
    assert (val == 0xFF800000).all()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("kind,kw", [("constant", {}), ("levels", {"levels": 4}),
                                     ("specials", {"fraction": 0.02})])
def test_ties_and_specials_across_pieces(dtype, kind, kw):
    N, k = 2_500_000, 700
    bits, _ = workloads.generate(1, N, dtype, kind, seed=63, **kw)
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    assert_same(*long_row(bits, dtype, k, 1024, 1024), ref_idx, ref_val)


def test_result_does_not_depend_on_the_seed():
    bits, _ = workloads.generate(1, 3_000_000, "bf16", "gumbel_spikes", seed=64, spikes=300)
    ref_idx, ref_val = oracle.topk(bits, "bf16", 50)
    for seed in (1, 2, 0xDEADBEEF):
        assert_same(*long_row(bits, "bf16", 50, 1024, 1024, seed=seed), ref_idx, ref_val)


def test_same_result_as_the_matrix_entry_point():
    bits, _ = workloads.generate(1, 1 << 21, "fp32", "ascending", seed=65)
    x = to_device(bits, "fp32")
    i1, v1 = ds.topk(x, 300, 1024, 1024)
    i2, v2 = ds.topk_long_row(x.reshape(-1), 300, 1024, 1024)
    torch.cuda.synchronize()
    assert torch.equal(i1[0], i2) and torch.equal(v1[0].view(torch.int32), v2.view(torch.int32))


def test_short_row_is_selected_directly():
    # too short to cut: no workspace, the row goes to the matrix kernel
    N, k = 50_000, 1024
    nb, P, G = plan("fp32", N, k, 1024, 1024)
    assert (nb, P, G) == (0, N, 1)
    bits, _ = workloads.generate(1, N, "fp32", "normal", seed=66)
    x = to_device(bits.reshape(-1), "fp32")
    out_i = torch.empty(k, dtype=torch.int32, device=DEV)
    out_v = torch.empty(k, dtype=torch.float32, device=DEV)
    ds.ds_topk_long_row(x.data_ptr(), 0, N, k, 1024, 1024, SEED, None, 0, out_i.data_ptr(),
                        out_v.data_ptr(), None)
    torch.cuda.synchronize()
    ref_idx, ref_val = oracle.topk(bits, "fp32", k)
    assert_same(out_i.cpu().numpy()[None], val_bits(out_v, "fp32")[None], ref_idx, ref_val)


def test_workspace_is_checked():
    N, k = 4_000_000, 256
    nb, P, G = plan("fp32", N, k, 1024, 1024)
    assert G > 1 and nb > 0
    x = torch.zeros(N, dtype=torch.float32, device=DEV)
    ws = torch.empty(nb + 256, dtype=torch.uint8, device=DEV)
    out_i = torch.empty(k, dtype=torch.int32, device=DEV)
    out_v = torch.empty(k, dtype=torch.float32, device=DEV)
    args = (x.data_ptr(), 0, N, k, 1024, 1024, SEED)
    outs = (out_i.data_ptr(), out_v.data_ptr(), None)
    for ptr, size in [(None, nb), (ws.data_ptr(), nb - 1), (ws.data_ptr() + 16, nb)]:
        with pytest.raises(ds.DSError) as e:
            ds.ds_topk_long_row(*args, ptr, size, *outs)
        assert e.value.status == ds.DS_EINVAL
    ds.ds_topk_long_row(*args, ws.data_ptr(), nb, *outs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_i.cpu().numpy(), np.arange(k))


def test_long_row_workload_full_size():
    """The benchmarked long-row workload, checked by properties at full size:
    values equal torch.topk's, every value is x[idx], and the index set is
    exactly {j : x_j > v_k} plus the lowest-index elements equal to v_k."""
    c = workloads.LONG_ROW
    bits, _ = workloads.generate(1, c["N"], c["dtype"], c["kind"], c["seed"])
    x = to_device(bits.reshape(-1), c["dtype"])
    del bits
    idx, val = ds.topk_long_row(x, c["k"], c["B"], c["B2"])
    ref = torch.topk(x, c["k"], largest=True, sorted=True).values
    torch.cuda.synchronize()
    assert torch.equal(val, ref)
    assert torch.equal(x[idx.long()], val)
    assert len(torch.unique(idx)) == c["k"]
    vk, ik = val[-1], idx[-1]
    j = torch.arange(x.numel(), device=DEV)
    chosen = (x > vk) | ((x == vk) & (j <= ik))
    assert int(chosen.sum()) == c["k"]
    assert bool(chosen[idx.long()].all())
    # order: value descending, ties by lower index
    assert bool((val[:-1] >= val[1:]).all())
    tie = val[:-1] == val[1:]
    assert bool((idx[:-1][tie] < idx[1:][tie]).all())


def topk_set_is_exact(x, idx, val, k):
    """The outputs are exactly the row's top k under the total order (no NaN
    or signed zero among the top values here): values are x[idx] and sorted,
    indices are distinct, and #{x > v_k} + #{x == v_k, index <= i_k} == k."""
    assert torch.equal(x[idx.long()], val)
    assert len(torch.unique(idx)) == k
    f = val.float()
    assert bool((f[:-1] >= f[1:]).all())
    tie = f[:-1] == f[1:]
    assert bool((idx[:-1][tie] < idx[1:][tie]).all())
    vk, ik = val[-1], int(idx[-1])
    n_gt = int((x > vk).sum())
    n_eq = int((x[:ik + 1] == vk).sum())
    assert n_gt + n_eq == k


def device_normal_bf16(n, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    x = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        x[s:e] = torch.randn(e - s, generator=g, device=DEV).to(torch.bfloat16)
    return x


def test_long_row_at_the_index_limit():
    # N = 2^31 - 1 bf16 (4 GB): row indices up to 2^31 - 2 from piece * P + local
    N, k = (1 << 31) - 1, 256
    _, P, G = plan("bf16", N, k, 4096, 4096)
    assert G > 1 and (G - 1) * P < N
    x = device_normal_bf16(N, seed=67)
    idx, val = ds.topk_long_row(x, k, 4096, 4096)
    torch.cuda.synchronize()
    topk_set_is_exact(x, idx, val, k)


def test_matrix_rows_beyond_2_31_elements():
    # 4200 rows of 2^19 bf16: rows from 4096 on start past element 2^31
    rows, N, k = 4200, 1 << 19, 128
    x = device_normal_bf16(rows * N, seed=68).view(rows, N)
    idx, val = ds.topk(x, k, 1024, 1024)
    ref = torch.topk(x, k, dim=-1, largest=True, sorted=True).values
    torch.cuda.synchronize()
    assert torch.equal(val, ref)
    for r in (0, 4095, 4096, rows - 1):
        topk_set_is_exact(x[r], idx[r], val[r], k)


def test_refused_second_launch_enqueues_nothing():
    # B = 16 makes 2048 pieces; their 2048 * 600 results are more blocks per
    # slice than the second launch takes.  The call is refused before either
    # launch: workspace and outputs keep what they held.
    N, k, B = 1 << 27, 600, 16
    nb, P, G = plan("fp32", N, k, B, B)
    assert G * k // B > 16 * 4096
    x = torch.zeros(N, dtype=torch.float32, device=DEV)
    ws = torch.full((nb,), 0x5A, dtype=torch.uint8, device=DEV)
    oi = torch.full((k,), -7, dtype=torch.int32, device=DEV)
    ov = torch.full((k,), 3.0, dtype=torch.float32, device=DEV)
    with pytest.raises(ds.DSError) as e:
        ds.ds_topk_long_row(x.data_ptr(), 0, N, k, B, B, SEED, ws.data_ptr(), nb, oi.data_ptr(),
                            ov.data_ptr(), None)
    assert e.value.status == ds.DS_EUNSUPPORTED
    torch.cuda.synchronize()
    assert bool((ws == 0x5A).all()) and bool((oi == -7).all()) and bool((ov == 3.0).all())
