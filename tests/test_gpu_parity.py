"""GPU parity: the CUDA library against the CPU oracle, bit for bit.

Every result of the library is unique (value descending, NaN above +inf,
-0 == +0, ties by lower index), so indices and value bits must equal the
oracle's exactly.  The instrumented counters (A, R, W, peak) must equal the
step-by-step model's for the same block order, which also checks that both
sides draw the same Philox permutation.
"""
import ctypes

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


def to_device(bits, dtype):
    if dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(DEV).view(torch.float32)
    t16 = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(t16)


def val_bits(t, dtype):
    if dtype == "fp32":
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def float_bits(f, dtype):
    """Bit patterns of float32 values in `dtype` (round to nearest even)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    if dtype == "fp32":
        return f.view(np.uint32).copy()
    return workloads.to_bf16_bits(f) if dtype == "bf16" else workloads.to_f16_bits(f)


def run(bits, dtype, k, B, B2, seed=SEED, row_len=None, splits=0, stats=False):
    x = to_device(bits, dtype)
    rl = None if row_len is None else torch.from_numpy(np.asarray(row_len, np.int32)).to(DEV)
    out = ds.topk(x, k, B, B2, seed=seed, row_len=rl, splits=splits, stats=stats)
    torch.cuda.synchronize()
    res = [out[0].cpu().numpy(), val_bits(out[1], dtype)]
    if stats:
        res.append(out[2].cpu().numpy())
    return res


def assert_same(got_idx, got_val, ref_idx, ref_val):
    bad = np.nonzero((got_idx != ref_idx).any(axis=1) | (got_val != ref_val).any(axis=1))[0]
    assert len(bad) == 0, "rows differ from the oracle: %s (first: idx %s vs %s)" % (
        bad[:8].tolist(), got_idx[bad[0]][:8].tolist(), ref_idx[bad[0]][:8].tolist())


_cache = {}


def config_case(name):
    if name not in _cache:
        c = workloads.CONFIGS[name]
        bits, row_len = workloads.config_inputs(name)
        ref = oracle.topk(bits, c["dtype"], c["k"], row_len=row_len)
        _cache[name] = (c, bits, row_len, ref)
    return _cache[name]


# ---------------------------------------------------------------------------
# The five workloads at full size, automatic plan and one CTA per row.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
@pytest.mark.parametrize("splits", [0, 1])
def test_workload_parity(name, splits):
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    idx, val = run(bits, c["dtype"], c["k"], c["B"], c["B2"], row_len=row_len, splits=splits)
    assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("name", ["dsa_index_bf16", "adversarial_fp32", "small_fp32",
                                  "dsa_decode_ragged_fp32"])
@pytest.mark.parametrize("splits", [2, 3, 8, 16])
def test_workload_parity_forced_splits(name, splits):
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    try:
        idx, val = run(bits, c["dtype"], c["k"], c["B"], c["B2"], row_len=row_len, splits=splits)
    except ds.DSError as e:
        assert e.status == ds.DS_EUNSUPPORTED   # merge buffer too large for shared memory
        pytest.skip(str(e))
    assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("name", ["dsa_index_bf16", "adversarial_fp32"])
def test_result_is_seed_invariant(name):
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    for seed in [0, 1, 2, 3, 0xFFFFFFFF, 1 << 40, 0x123456789ABCDEF, 2 ** 64 - 1]:
        idx, val = run(bits, c["dtype"], c["k"], c["B"], c["B2"], seed=seed, row_len=row_len)
        assert_same(idx, val, ref_idx, ref_val)


# ---------------------------------------------------------------------------
# Counters: GPU == step-by-step model for the same seed and split factor.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
@pytest.mark.parametrize("splits", [1, 4])
def test_stats_match_model(name, splits):
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    for seed in [SEED, 12345]:
        m_idx, m_val, m_stats = oracle.model(bits, c["dtype"], c["k"], c["B"], c["B2"], seed,
                                             row_len=row_len, splits=splits)
        idx, val, st = run(bits, c["dtype"], c["k"], c["B"], c["B2"], seed=seed,
                           row_len=row_len, splits=splits, stats=True)
        assert_same(idx, val, ref_idx, ref_val)
        mism = np.nonzero((st != m_stats).any(axis=2))
        assert len(mism[0]) == 0, "stats differ at (row, slice) %s: gpu %s model %s" % (
            list(zip(mism[0][:4], mism[1][:4])), st[mism][:4].tolist(), m_stats[mism][:4].tolist())
        A, R, W, peak = (st[..., i] for i in range(4))
        assert np.all(W == A + c["k"] * R)
        assert np.all(peak <= c["k"] + c["B2"] + c["B"] - 1)


def test_identity_order_blows_up_the_work_on_ascending_rows():
    """DeepSelect-deep-dive, "算法": the block order must be random and
    independent of the data.  On the adversarial workload's ascending rows,
    index order (ds_topk_stats_order) makes every block beat the threshold:
    every element is appended and W is many times the random order's.  Both
    orders' counters equal the step-by-step model's for the same order, and
    the result is the oracle's either way."""
    c = workloads.CONFIGS["adversarial_fp32"]
    bits, _ = workloads.config_inputs("adversarial_fp32")
    bits = np.ascontiguousarray(bits[:16])  # rows 0..15: sorted ascending
    k, B, B2 = c["k"], c["B"], c["B2"]
    ref_idx, ref_val = oracle.topk(bits, "fp32", k)
    x = to_device(bits, "fp32")
    W = {}
    for order in (ds.DS_ORDER_RANDOM, ds.DS_ORDER_IDENTITY):
        out = ds.topk(x, k, B, B2, seed=SEED, splits=1, stats=True, order=order)
        torch.cuda.synchronize()
        idx, val, st = out[0].cpu().numpy(), val_bits(out[1], "fp32"), out[2].cpu().numpy()
        assert_same(idx, val, ref_idx, ref_val)
        _, _, m_stats = oracle.model(bits, "fp32", k, B, B2, SEED, splits=1,
                                     identity_order=order == ds.DS_ORDER_IDENTITY)
        np.testing.assert_array_equal(st, m_stats)
        W[order] = st[:, 0, 2]
    n = bits.shape[1]
    A_id = st[:, 0, 0]
    assert np.all(A_id == n)  # index order on ascending rows: every element is appended
    assert np.all(W[ds.DS_ORDER_IDENTITY] >= 10 * W[ds.DS_ORDER_RANDOM])


# ---------------------------------------------------------------------------
# Edge cases.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("kind", ["specials", "levels", "constant", "ascending"])
def test_ties_and_special_values(dtype, kind):
    bits, _ = workloads.generate(16, 20000, dtype, kind, seed=17, fraction=0.2, value=0.0)
    for k, B, B2, splits in [(100, 256, 256, 0), (1, 64, 64, 1), (777, 512, 128, 3),
                             (5000, 1024, 1024, 1)]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k)
        idx, val = run(bits, dtype, k, B, B2, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)
    # k = N: the whole row in order
    short = np.ascontiguousarray(bits[:, :3000])
    ref_idx, ref_val = oracle.topk(short, dtype, 3000)
    idx, val = run(short, dtype, 3000, 512, 512, splits=1)
    assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("kind", ["normal", "specials", "levels", "constant", "ascending"])
def test_first_threshold_for_large_k(dtype, kind):
    # k above 128 starts from a threshold taken from the chunk maxima of each
    # warp's first stages (one range histogram): k on both sides of every
    # group count (1, 2, 4, 8, 16 groups per lane), small blocks that leave
    # lanes without chunks, ragged rows around k + B2, ties at the bin edge
    bits, _ = workloads.generate(6, 40000, dtype, kind, seed=43, fraction=0.3, value=0.5)
    row_len = np.array([40000, 39999, 5000, 3000, 1200, 20000], dtype=np.int32)
    for k, B, B2, splits in [(129, 1024, 64, 1), (256, 64, 64, 1), (257, 512, 256, 0),
                             (512, 1024, 128, 1), (513, 64, 512, 2), (1024, 1024, 256, 1),
                             (1025, 256, 1024, 3), (2048, 1024, 64, 1), (2049, 512, 512, 1),
                             (4096, 1024, 1024, 1)]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k, row_len=row_len)
        idx, val = run(bits, dtype, k, B, B2, row_len=row_len, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("kind", ["normal", "specials", "levels", "ascending"])
def test_split_rows_with_a_large_union(dtype, kind):
    # splits * k above 8192: one radix select over the union of the slices'
    # candidates, its histograms summed across the cluster, then CTA 0
    # orders the k selected entries; ragged rows leave some slices short or
    # empty, odd split counts included
    bits, _ = workloads.generate(6, 60000, dtype, kind, seed=29, fraction=0.2, value=0.0)
    row_len = np.array([60000, 0, 1500, 4095, 33333, 59999], dtype=np.int32)
    for k, B, B2, splits in [(1100, 512, 512, 8), (1300, 1024, 256, 7), (2000, 512, 1024, 5),
                             (4096, 1024, 1024, 3), (5000, 1024, 1024, 2)]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k, row_len=row_len)
        idx, val = run(bits, dtype, k, B, B2, row_len=row_len, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("kind", ["normal", "constant", "levels", "specials", "ascending"])
def test_split_rows_select_across_the_cluster_or_pruned(dtype, kind):
    # 6144 < splits * k <= 8192: the select across the cluster; k above
    # 6144: slices send CTA 0 only entries at or above the largest slice
    # k-th composite (ties across slices, short and empty slices included)
    bits, _ = workloads.generate(5, 50000, dtype, kind, seed=37, fraction=0.2, value=-1.5)
    row_len = np.array([50000, 0, 900, 7000, 49999], dtype=np.int32)
    for k, B, B2, splits in [(900, 512, 512, 7), (1024, 1024, 512, 8), (1600, 256, 1024, 4),
                             (6500, 512, 512, 2)]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k, row_len=row_len)
        idx, val = run(bits, dtype, k, B, B2, row_len=row_len, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("kind,rows,N,k,B,B2", [("normal", 64, 32768, 512, 1024, 1024),
                                                ("gumbel_spikes", 16, 128000, 50, 1024, 1024),
                                                ("adversarial", 8, 65536, 1024, 1024, 1024)])
@pytest.mark.parametrize("splits", [0, 1])
def test_fp16_workload_shapes(kind, rows, N, k, B, B2, splits):
    # the DSA index, sampling and adversarial shapes with IEEE fp16 inputs
    bits, _ = workloads.generate(rows, N, "fp16", kind, seed=31)
    ref_idx, ref_val = oracle.topk(bits, "fp16", k)
    idx, val = run(bits, "fp16", k, B, B2, splits=splits)
    assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("kind", ["normal", "levels", "specials"])
def test_output_orderings_of_every_size(dtype, kind):
    # k on both sides of every ordering strategy: counting ranks (<= 256),
    # ranks across warp runs (<= 1024), merge-path sort (<= 2048), shared-
    # memory bitonic (above), with one CTA per row and with splits
    bits, _ = workloads.generate(4, 12000, dtype, kind, seed=41, fraction=0.1)
    for k in [255, 256, 257, 512, 513, 1024, 1025, 1500, 2048, 2049, 3000]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k)
        for splits in [1, 2]:
            idx, val = run(bits, dtype, k, 1024, 1024, splits=splits)
            assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_negative_zero_and_nan_bits_are_returned_as_read(dtype):
    f = np.zeros((4, 3000), dtype=np.float32)
    f[:, ::2] = -0.0
    f[1, 100:110] = np.nan
    f[2, 5] = -np.inf
    f[3, :] = -1.0
    f[3, 2999] = -0.0
    bits = float_bits(f, dtype)
    if dtype == "fp32":
        bits[1, 100:110] |= np.arange(1, 11, dtype=np.uint32)      # NaN payloads
        bits[1, 105] |= np.uint32(0x80000000)                      # a negative NaN
    if dtype == "fp16":
        bits[1, 100:110] = np.uint16(0x7C00) | np.arange(1, 11, dtype=np.uint16)
        bits[1, 105] |= np.uint16(0x8000)
    for k in [1, 17, 64]:
        ref_idx, ref_val = oracle.topk(bits, dtype, k)
        idx, val = run(bits, dtype, k, 128, 128, splits=1)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_row_len_edges(dtype):
    bits, _ = workloads.generate(8, 4096, dtype, "normal", seed=23)
    row_len = np.array([0, 1, 63, 64, 65, 4096, 100000, -7], dtype=np.int32)
    for splits in [0, 1, 4, 16]:
        ref_idx, ref_val = oracle.topk(bits, dtype, 64, row_len=row_len)
        idx, val = run(bits, dtype, 64, 128, 128, row_len=row_len, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("N,k,B,B2", [(1, 1, 1, 1), (7, 3, 1, 1), (1000, 1000, 100, 3),
                                      (4099, 13, 100, 50), (3001, 200, 1000, 17),
                                      (65536, 64, 16384, 512), (20000, 2048, 64, 4000)])
def test_shapes_block_sizes_and_plain_load_path(dtype, N, k, B, B2):
    """Odd N and B take the plain-load path; others the bulk-copy path."""
    bits, _ = workloads.generate(5, N, dtype, "normal", seed=N + k)
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    for splits in [0, 1, 2]:
        idx, val = run(bits, dtype, k, B, B2, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_misaligned_input_pointer(dtype):
    rows, N, k = 6, 8192, 100
    bits, _ = workloads.generate(rows, N, dtype, "normal", seed=31)
    esz = 4 if dtype == "fp32" else 2
    flat = np.zeros(rows * N + 8, dtype=bits.dtype)
    flat[1:1 + rows * N] = bits.ravel()
    xt = to_device(flat, dtype)
    out_idx = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    out_val = torch.empty((rows, k), dtype=xt.dtype, device=DEV)
    code = {"fp32": ds.DS_FP32, "bf16": ds.DS_BF16, "fp16": ds.DS_FP16}[dtype]
    plan = ds.ds_topk_plan(xt.data_ptr() + esz, code, rows, N, k, 256, 256, 1)
    assert plan["async_copy"] == 0
    ds.ds_topk_ex(xt.data_ptr() + esz, code, rows, None, N, k, 256, 256, 7, 1,
                  out_idx.data_ptr(), out_val.data_ptr(), None, None)
    torch.cuda.synchronize()
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    assert_same(out_idx.cpu().numpy(), val_bits(out_val, dtype), ref_idx, ref_val)


def test_largest_k_that_fits():
    # ds_topk_max_k assumes the longest row the block order allows: N = 4096 B
    kmax = ds.ds_topk_max_k(ds.DS_FP32, 1024, 1024)
    assert kmax > 2048
    N = 1024 * 4096
    bits, _ = workloads.generate(1, N, "fp32", "normal", seed=5)
    ref_idx, ref_val = oracle.topk(bits, "fp32", kmax)
    idx, val = run(bits, "fp32", kmax, 1024, 1024, splits=1)
    assert_same(idx, val, ref_idx, ref_val)
    with pytest.raises(ds.DSError) as e:
        run(bits, "fp32", kmax + 1, 1024, 1024, splits=1)
    assert e.value.status == ds.DS_EUNSUPPORTED


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_one_long_row(dtype):
    # 2^25 elements in one row: sixteen slices of one cluster
    bits, _ = workloads.generate(1, 1 << 25, dtype, "gumbel_spikes", seed=43, spikes=64)
    ref_idx, ref_val = oracle.topk(bits, dtype, 100)
    idx, val = run(bits, dtype, 100, 4096, 4096)
    assert_same(idx, val, ref_idx, ref_val)
    # the block order of a slice holds at most 4096 blocks: a small B is refused
    # with a message, not run wrong
    with pytest.raises(ds.DSError):
        run(bits, dtype, 100, 256, 256)


def test_many_short_rows():
    # thousands of rows: many waves of one-CTA-per-row launches
    bits, row_len = workloads.generate(6000, 700, "bf16", "ragged_normal", seed=47, min_len=1)
    ref_idx, ref_val = oracle.topk(bits, "bf16", 16, row_len=row_len)
    idx, val = run(bits, "bf16", 16, 128, 128, row_len=row_len)
    assert_same(idx, val, ref_idx, ref_val)


def test_poisoned_tail_is_never_read():
    """Past row_len the input holds NaN, which would win every comparison."""
    bits, row_len = workloads.generate(16, 50000, "fp32", "ragged_normal", seed=8, min_len=1)
    cols = np.arange(50000)[None, :]
    bits[cols >= row_len[:, None]] = np.uint32(0x7FC00000)
    for splits in [0, 1, 5]:
        ref_idx, ref_val = oracle.topk(bits, "fp32", 300, row_len=row_len)
        idx, val = run(bits, "fp32", 300, 1000, 1000, row_len=row_len, splits=splits)
        assert_same(idx, val, ref_idx, ref_val)


def test_non_default_stream_and_zero_rows():
    c, bits, row_len, (ref_idx, ref_val) = config_case("dsa_index_bf16")
    x = to_device(bits, "bf16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx, val = ds.topk(x, c["k"], c["B"], c["B2"], stream=s)
    s.synchronize()
    assert_same(idx.cpu().numpy(), val_bits(val, "bf16"), ref_idx, ref_val)
    ds.ds_topk(x.data_ptr(), ds.DS_BF16, 0, None, c["N"], c["k"], c["B"], c["B2"], 0,
               idx.data_ptr(), val.data_ptr(), None)


@pytest.mark.parametrize("name", ["dsa_index_bf16", "dsa_decode_ragged_fp32"])
def test_host_buffer_entry_point(name):
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    rows, N, k = c["rows"], c["N"], c["k"]
    tdt = torch.float32 if c["dtype"] == "fp32" else torch.bfloat16
    x_host = torch.from_numpy(bits.view(np.int32 if c["dtype"] == "fp32" else np.int16)).pin_memory()
    rl_host = None if row_len is None else torch.from_numpy(row_len).pin_memory()
    oi_host = torch.empty((rows, k), dtype=torch.int32).pin_memory()
    ov_host = torch.empty((rows, k), dtype=x_host.dtype).pin_memory()
    x_dev = torch.empty((rows, N), dtype=tdt, device=DEV)
    rl_dev = None if row_len is None else torch.empty(rows, dtype=torch.int32, device=DEV)
    oi_dev = torch.empty((rows, k), dtype=torch.int32, device=DEV)
    ov_dev = torch.empty((rows, k), dtype=tdt, device=DEV)
    code = ds.DS_FP32 if c["dtype"] == "fp32" else ds.DS_BF16
    for _ in range(2):
        ds.ds_topk_host(x_host.data_ptr(), code, rows, None if rl_host is None else rl_host.data_ptr(),
                        N, k, c["B"], c["B2"], SEED, oi_host.data_ptr(), ov_host.data_ptr(),
                        x_dev.data_ptr(), None if rl_dev is None else rl_dev.data_ptr(),
                        oi_dev.data_ptr(), ov_dev.data_ptr(), None)
        got_val = ov_host.numpy().view(np.uint32 if c["dtype"] == "fp32" else np.uint16)
        assert_same(oi_host.numpy(), got_val, ref_idx, ref_val)


@pytest.mark.parametrize("name", ["dsa_index_bf16", "small_fp32"])
def test_host_async_entry_point_on_two_streams(name):
    # consecutive enqueue-only calls on two streams with two staging sets,
    # every result read back on the host after its stream completes
    c, bits, row_len, (ref_idx, ref_val) = config_case(name)
    rows, N, k = c["rows"], c["N"], c["k"]
    tdt = torch.float32 if c["dtype"] == "fp32" else torch.bfloat16
    x_host = torch.from_numpy(bits.view(np.int32 if c["dtype"] == "fp32" else np.int16)).pin_memory()
    code = ds.DS_FP32 if c["dtype"] == "fp32" else ds.DS_BF16
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    sets = [dict(oi_host=torch.empty((rows, k), dtype=torch.int32).pin_memory(),
                 ov_host=torch.empty((rows, k), dtype=x_host.dtype).pin_memory(),
                 x_dev=torch.empty((rows, N), dtype=tdt, device=DEV),
                 oi_dev=torch.empty((rows, k), dtype=torch.int32, device=DEV),
                 ov_dev=torch.empty((rows, k), dtype=tdt, device=DEV)) for _ in range(2)]
    for i in range(6):
        b = sets[i % 2]
        b["oi_host"].fill_(-7)
        ds.ds_topk_host_async(x_host.data_ptr(), code, rows, None, N, k, c["B"], c["B2"], SEED + i,
                              b["oi_host"].data_ptr(), b["ov_host"].data_ptr(), b["x_dev"].data_ptr(),
                              None, b["oi_dev"].data_ptr(), b["ov_dev"].data_ptr(),
                              streams[i % 2].cuda_stream)
        if i > 0:
            p = sets[(i - 1) % 2]
            streams[(i - 1) % 2].synchronize()
            got_val = p["ov_host"].numpy().view(np.uint32 if c["dtype"] == "fp32" else np.uint16)
            assert_same(p["oi_host"].numpy(), got_val, ref_idx, ref_val)
    torch.cuda.synchronize()


def test_plans_of_the_workloads():
    for name in workloads.CONFIG_ORDER:
        c = workloads.CONFIGS[name]
        code = ds.DS_FP32 if c["dtype"] == "fp32" else ds.DS_BF16
        plan = ds.ds_topk_plan(1 << 20, code, c["rows"], c["N"], c["k"], c["B"], c["B2"], 0)
        assert plan["async_copy"] == 1
        # calls without counters take the free-running kernel; its buffer
        # holds k + B2 plus one warp stage (2 KiB of elements)
        assert plan["kernel"] == 1
        esz = 4 if c["dtype"] == "fp32" else 2
        assert plan["capacity"] >= c["k"] + c["B2"] + 2048 // esz
        assert plan["grid"] == c["rows"] * plan["splits"]
        s = plan["splits"]
        assert s & (s - 1) == 0 and s <= 16
        # one wave: at most the resident CTAs of the device
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert plan["grid"] <= sms * plan["ctas_per_sm"]
        if sms == 152:
            # rows under 128 KiB stay whole (slices keep 64 KiB); long rows
            # fill two CTAs per SM
            want = {"small_fp32": 1, "dsa_index_bf16": 1, "dsa_decode_ragged_fp32": 8,
                    "sampling_logits_bf16": 1, "adversarial_fp32": 8}
            if name in want:
                assert s == want[name], (name, plan)
