"""The two-level selection behind ds_topk_long_row, checked on the CPU with
the oracle alone (no CUDA): cut the row into pieces of P elements, take every
piece's top k, take the top k of the piece results laid end to end, and map
each chosen position q to the row index (q // k) * P + (index within piece).
Under the total order (value descending, ties by lower index) this must be
the row's own top k -- including ties across pieces, NaN and signed zeros,
and a last piece shorter than k whose -inf pads tie with real -inf values.
"""
import numpy as np
import pytest

import oracle
import workloads

NEG_INF = {"fp32": np.uint32(0xFF800000), "bf16": np.uint16(0xFF80), "fp16": np.uint16(0xFC00)}


def two_level(bits, dtype, k, P, reverse_pieces=False):
    N = bits.shape[1]
    G = -(-N // P)
    pieces = np.full((G, P), NEG_INF[dtype], dtype=bits.dtype)
    pieces.reshape(-1)[:N] = bits[0]
    row_len = np.array([min(P, N - g * P) for g in range(G)], dtype=np.int32)
    idx1, val1 = oracle.topk(pieces, dtype, k, row_len=row_len)
    order = np.arange(G)[::-1] if reverse_pieces else np.arange(G)
    flat_val = val1[order].reshape(1, G * k)
    flat_idx = (idx1[order] + np.where(idx1[order] >= 0, order[:, None] * P, 0)).reshape(-1)
    q, v2 = oracle.topk(flat_val, dtype, k)
    return flat_idx[q[0]][None, :], v2


CASES = [
    ("fp32", "normal", {}, 10007, 64, 256),
    ("bf16", "levels", {"levels": 5}, 5000, 100, 128),
    ("bf16", "specials", {"fraction": 0.3}, 3001, 70, 96),
    ("fp16", "specials", {"fraction": 0.3}, 3001, 70, 96),
    ("fp32", "constant", {"value": 2.0}, 2049, 33, 64),
]


@pytest.mark.parametrize("dtype,kind,kw,N,k,P", CASES)
def test_two_level_selection_is_the_rows_top_k(dtype, kind, kw, N, k, P):
    bits, _ = workloads.generate(1, N, dtype, kind, seed=81, **kw)
    ref_idx, ref_val = oracle.topk(bits, dtype, k)
    idx, val = two_level(bits, dtype, k, P)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_array_equal(val, ref_val)


def test_short_last_piece_pads_never_win():
    # every element -inf and a last piece of one element: pads tie with the
    # real values and must lose to all of them
    k, P = 16, 64
    N = 5 * P + 1
    bits = np.full((1, N), NEG_INF["fp32"], dtype=np.uint32)
    idx, val = two_level(bits, "fp32", k, P)
    np.testing.assert_array_equal(idx[0], np.arange(k))
    assert (val == NEG_INF["fp32"]).all()


def test_piece_order_matters_for_ties():
    # negative control: laying the piece results out in reverse row order
    # breaks the tie order, so the check above has the power to see it
    bits, _ = workloads.generate(1, 4000, "bf16", "levels", seed=82, levels=3)
    ref_idx, _ = oracle.topk(bits, "bf16", 200)
    idx, _ = two_level(bits, "bf16", 200, 256, reverse_pieces=True)
    assert not np.array_equal(idx, ref_idx)
