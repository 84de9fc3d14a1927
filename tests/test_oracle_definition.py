"""Pins for the oracle's definition of top-k (CPU only).

The oracle is checked against things other than itself:
  * the worked example printed on milkfeng.top "CUDA 算子笔记 4",
    section "Top K Selection";
  * a brute-force rank count written from float semantics (not from the
    oracle's bit-level key map), exhaustive over short arrays of special
    values;
  * closed forms and library routines: numpy lexsort for k = len, numpy
    argmax for k = 1, constant / ascending / few-level rows;
  * the key map itself against numpy float comparisons, exhaustively for bf16.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF_F32 = np.uint32(0xFF800000)
NEG_INF_BF16 = np.uint16(0xFF80)
NEG_INF_F16 = np.uint16(0xFC00)


def _read_golden(name):
    fields = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, value = line.partition(":")
            fields[key.strip()] = value.split()
    return fields


def test_worked_example_from_page():
    g = _read_golden("topk_worked_example.txt")
    values = np.array([float(v) for v in g["input"]], dtype=np.float32)
    k = int(g["k"][0])
    expected = np.array([float(v) for v in g["output"]], dtype=np.float32)
    idx, val = oracle.topk(values[None, :], "fp32", k)
    np.testing.assert_array_equal(val[0].view(np.float32), expected)
    # indices: the position of each printed output value in the input
    np.testing.assert_array_equal(idx[0], [int(np.nonzero(values == v)[0][0]) for v in expected])
    # bf16 gives the same answer for these exactly representable values
    idx16, val16 = oracle.topk(workloads.to_bf16_bits(values[None, :]), "bf16", k)
    np.testing.assert_array_equal(idx16, idx)
    np.testing.assert_array_equal(workloads.bits_to_f32(val16, "bf16")[0], expected)


# ---------------------------------------------------------------------------
# Brute force: i is selected at output position p iff exactly p elements come
# before it, where "j comes before i" is defined with Python floats:
# NaN above everything (NaNs equal), -0 == +0, then lower index first.
# ---------------------------------------------------------------------------
ALPHABET = [-math.inf, -1.0, -0.0, 0.0, 1.0, 2.0, math.inf, math.nan, -math.nan]


def _before(a, ia, b, ib):
    """True if value a at index ia comes before value b at index ib."""
    na, nb = math.isnan(a), math.isnan(b)
    if na and nb:
        return ia < ib
    if na != nb:
        return na
    if a != b:
        return a > b
    return ia < ib


def _brute_force_order(values):
    n = len(values)
    ranks = [sum(_before(values[j], j, values[i], i) for j in range(n)) for i in range(n)]
    order = [None] * n
    for i, r in enumerate(ranks):
        order[r] = i
    return order


def _vectorised_ranks(f):
    """Same rank count as _brute_force_order, for a batch [rows, n] (numpy)."""
    rows, n = f.shape
    a = f[:, :, None]      # candidate j
    b = f[:, None, :]      # element i
    na, nb = np.isnan(a), np.isnan(b)
    j_idx = np.arange(n)[None, :, None]
    i_idx = np.arange(n)[None, None, :]
    with np.errstate(invalid="ignore"):
        greater = (a > b) & ~na & ~nb
        equal = ((a == b) & ~na & ~nb) | (na & nb)
    before = (na & ~nb) | greater | (equal & (j_idx < i_idx))
    return before.sum(axis=1)  # [rows, n]: rank of element i


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_bruteforce_exhaustive_specials(dtype, n):
    combos = np.array(list(itertools.product(range(len(ALPHABET)), repeat=n)), dtype=np.int64)
    f = np.array(ALPHABET, dtype=np.float32)[combos]
    bits = f.view(np.uint32) if dtype == "fp32" else \
        workloads.to_bf16_bits(f) if dtype == "bf16" else workloads.to_f16_bits(f)
    ranks = _vectorised_ranks(f)
    expected_order = np.argsort(ranks, axis=1)   # ranks are a permutation of 0..n-1
    for k in sorted({1, (n + 1) // 2, n}):
        idx, val = oracle.topk(bits, dtype, k)
        np.testing.assert_array_equal(idx, expected_order[:, :k])
        np.testing.assert_array_equal(val, np.take_along_axis(bits, expected_order[:, :k], axis=1))


def test_bruteforce_scalar_crosscheck():
    # the vectorised rank count above agrees with the scalar definition
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(1, 9))
        values = [ALPHABET[i] for i in rng.integers(0, len(ALPHABET), size=n)]
        f = np.array(values, dtype=np.float32)[None, :]
        assert list(np.argsort(_vectorised_ranks(f)[0])) == _brute_force_order(values)
        k = int(rng.integers(1, n + 1))
        idx, _ = oracle.topk(f, "fp32", k)
        assert list(idx[0]) == _brute_force_order(values)[:k]


def test_bruteforce_random_longer_rows():
    rng = np.random.default_rng(11)
    for n in [7, 9, 12, 17]:
        f = np.array(ALPHABET, dtype=np.float32)[rng.integers(0, len(ALPHABET), size=(400, n))]
        order = np.argsort(_vectorised_ranks(f), axis=1)
        for k in [1, 3, n]:
            idx, val = oracle.topk(f, "fp32", k)
            np.testing.assert_array_equal(idx, order[:, :k])


# ---------------------------------------------------------------------------
# Closed forms and library routines.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_k_equals_len_is_full_stable_descending_sort(dtype):
    bits, _ = workloads.generate(6, 3000, dtype, "normal", seed=3)
    f = workloads.bits_to_f32(bits, dtype)
    idx, val = oracle.topk(bits, dtype, 3000)
    for r in range(6):
        order = np.lexsort((np.arange(3000), -f[r]))   # value desc, then index asc
        np.testing.assert_array_equal(idx[r], order)
        np.testing.assert_array_equal(val[r], bits[r][order])


def test_k1_is_argmax_lowest_index_nan_first():
    bits, _ = workloads.generate(64, 500, "fp32", "specials", seed=4, fraction=0.02)
    f = bits.view(np.float32)
    idx, val = oracle.topk(bits, "fp32", 1)
    # numpy argmax returns the first NaN if any, else the first maximum
    np.testing.assert_array_equal(idx[:, 0], np.argmax(f, axis=1))
    np.testing.assert_array_equal(val[:, 0], bits[np.arange(64), idx[:, 0]])


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_constant_row_gives_first_k_indices(dtype):
    bits, _ = workloads.generate(3, 1000, dtype, "constant", seed=0, value=-3.5)
    idx, val = oracle.topk(bits, dtype, 77)
    np.testing.assert_array_equal(idx, np.tile(np.arange(77), (3, 1)))
    np.testing.assert_array_equal(val, bits[:, :77])


def test_ascending_distinct_row_gives_last_indices():
    bits, _ = workloads.generate(4, 5000, "fp32", "ascending", seed=8)
    f = bits.view(np.float32)
    assert all(len(np.unique(f[r])) == 5000 for r in range(4))
    idx, _ = oracle.topk(bits, "fp32", 300)
    np.testing.assert_array_equal(idx, np.tile(np.arange(4999, 4699, -1), (4, 1)))


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_few_levels_take_lowest_indices_of_top_levels(dtype):
    bits, _ = workloads.generate(5, 4000, dtype, "levels", seed=9, levels=16)
    f = workloads.bits_to_f32(bits, dtype)
    k = 700
    idx, _ = oracle.topk(bits, dtype, k)
    for r in range(5):
        expected = np.concatenate([np.nonzero(f[r] == lv)[0] for lv in range(15, -1, -1)])[:k]
        np.testing.assert_array_equal(idx[r], expected)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_row_len_padding_and_clamping(dtype):
    bits, _ = workloads.generate(5, 64, dtype, "normal", seed=12)
    row_len = np.array([0, 3, 64, 1000, -5], dtype=np.int32)
    idx, val = oracle.topk(bits, dtype, 10, row_len=row_len)
    full_idx, _ = oracle.topk(bits, dtype, 10)
    pad = {"fp32": NEG_INF_F32, "bf16": NEG_INF_BF16, "fp16": NEG_INF_F16}[dtype]
    assert (idx[0] == -1).all() and (val[0] == pad).all()
    short_idx, _ = oracle.topk(bits[1:2, :3], dtype, 3)
    np.testing.assert_array_equal(idx[1, :3], short_idx[0])
    assert (idx[1, 3:] == -1).all() and (val[1, 3:] == pad).all()
    np.testing.assert_array_equal(idx[2], full_idx[2])
    np.testing.assert_array_equal(idx[3], full_idx[3])          # clamped to N
    assert (idx[4] == -1).all()                                  # negative -> empty


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_output_invariants_random(dtype):
    bits, row_len = workloads.generate(12, 4096, dtype, "ragged_normal", seed=21, min_len=100)
    k = 256
    idx, val = oracle.topk(bits, dtype, k, row_len=row_len)
    f = workloads.bits_to_f32(bits, dtype)
    for r in range(12):
        n = min(k, int(row_len[r]))
        sel = idx[r, :n]
        assert len(set(sel.tolist())) == n and sel.min() >= 0 and sel.max() < row_len[r]
        np.testing.assert_array_equal(val[r, :n], bits[r, sel])
        v = f[r, sel]
        # sorted by (value desc, index asc)
        assert all((v[i] > v[i + 1]) or (v[i] == v[i + 1] and sel[i] < sel[i + 1])
                   for i in range(n - 1))
        # every unselected valid element is at or below the k-th
        rest = np.setdiff1d(np.arange(row_len[r]), sel)
        if len(rest):
            kth_v, kth_i = v[-1], sel[-1]
            assert np.all((f[r, rest] < kth_v) | ((f[r, rest] == kth_v) & (rest > kth_i)))


# ---------------------------------------------------------------------------
# Key map: unsigned order of keys == the total order on values.
# ---------------------------------------------------------------------------
def _check_sorted_by_key(f_sorted):
    a, b = f_sorted[:-1], f_sorted[1:]
    na, nb = np.isnan(a), np.isnan(b)
    with np.errstate(invalid="ignore"):
        ok = (nb & ~na) | (na & nb) | (~na & ~nb & (a <= b))
    assert ok.all()


def test_bf16_key_map_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = workloads.bits_to_f32(bits, "bf16")
    k = oracle.keys(bits, "bf16")
    assert k.max() <= 0xFFFF
    order = np.argsort(k, kind="stable")
    _check_sorted_by_key(f[order])
    ks = k[order]
    fs = f[order]
    same = ks[:-1] == ks[1:]
    # equal keys exactly when equal values (or both NaN)
    with np.errstate(invalid="ignore"):
        eq_val = (fs[:-1] == fs[1:]) | (np.isnan(fs[:-1]) & np.isnan(fs[1:]))
    np.testing.assert_array_equal(same, eq_val)
    # bf16 keys agree with fp32 keys of the exact widening
    k32 = oracle.keys(f.view(np.uint32), "fp32")
    np.testing.assert_array_equal(np.argsort(k, kind="stable"), np.argsort(k32, kind="stable"))


def test_fp16_key_map_exhaustive():
    # every IEEE binary16 pattern, ordered by key, is ordered by value (numpy
    # float16 compares), and keys are equal exactly for equal values
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = workloads.bits_to_f32(bits, "fp16")
    np.testing.assert_array_equal(f, bits.view(np.float16).astype(np.float32))
    k = oracle.keys(bits, "fp16")
    assert k.max() <= 0xFFFF
    order = np.argsort(k, kind="stable")
    h = bits.view(np.float16)[order]
    a, b = h[:-1], h[1:]
    na, nb = np.isnan(a), np.isnan(b)
    with np.errstate(invalid="ignore"):
        assert ((nb & ~na) | (na & nb) | (~na & ~nb & (a <= b))).all()
        same = k[order][:-1] == k[order][1:]
        np.testing.assert_array_equal(same, (a == b) | (na & nb))
    # the boundaries: +inf is the largest non-NaN key, -0 and +0 share a key
    inf_key = oracle.keys(np.array([0x7C00], np.uint16), "fp16")[0]
    assert inf_key == k[~np.isnan(bits.view(np.float16))].max()
    assert oracle.keys(np.array([0x8000, 0x0000], np.uint16), "fp16").tolist() == [0x8000, 0x8000]
    # fp16 keys order the values exactly as fp32 keys of the widening do
    k32 = oracle.keys(f.view(np.uint32), "fp32")
    np.testing.assert_array_equal(np.argsort(k, kind="stable"), np.argsort(k32, kind="stable"))


def test_fp32_key_map_exhaustive():
    """All 2^32 fp32 patterns (oracle sweep in C): walked in increasing
    numeric order as C floats compare them, the key increases with them,
    equal only at -0 -> +0; every NaN pattern maps to the largest key."""
    assert oracle.load().ds_oracle_sweep_f32() == 0


def test_fp32_key_map_sampled_and_edges():
    rng = np.random.default_rng(1)
    edges = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x807FFFFF, 0x00800000,
                      0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7F800001, 0xFFC00000,
                      0x7FFFFFFF, 0xFFFFFFFF, 0x3F800000, 0xBF800000], dtype=np.uint32)
    bits = np.concatenate([edges, rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64)
                           .astype(np.uint32)])
    f = bits.view(np.float32)
    k = oracle.keys(bits, "fp32")
    order = np.argsort(k, kind="stable")
    _check_sorted_by_key(f[order])
    ks, fs = k[order], f[order]
    with np.errstate(invalid="ignore"):
        eq_val = (fs[:-1] == fs[1:]) | (np.isnan(fs[:-1]) & np.isnan(fs[1:]))
    np.testing.assert_array_equal(ks[:-1] == ks[1:], eq_val)
