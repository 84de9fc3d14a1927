"""Pins for the step-by-step model of the DeepSelect loop (CPU only).

PFCCLab/DeepSelect "DeepSelect-deep-dive":
  * section "算法" -- the loop itself and its notes: the candidate buffer never
    holds more than k + B2 + B entries, and the loop returns the top-k;
  * section "RadixSelectTopK 总处理元素数的期望上界" -- W = A + kR, R*B2 <= A, and
    E[W] <= (1 + k/B2) (k + B + B2) H_m with m = ceil(N/B), the expectation
    taken over the random block order alone.
The model's output is compared with the oracle's plain definition, which is
itself pinned in test_oracle_definition.py.
"""
import math

import numpy as np
import pytest

import oracle
import workloads


def harmonic(m):
    return sum(1.0 / i for i in range(1, m + 1))


def w_bound(N, k, B, B2):
    m = -(-N // B)
    return (1.0 + k / B2) * (k + B + B2) * harmonic(m)


def check_identities(stats, k, B, B2):
    A, R, W, peak = stats[..., 0], stats[..., 1], stats[..., 2], stats[..., 3]
    np.testing.assert_array_equal(W, A + k * R)
    assert np.all(R * B2 <= A)
    assert np.all(peak <= k + B2 + B - 1)


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_model_matches_definition_on_every_workload(name):
    c = workloads.CONFIGS[name]
    bits, row_len = workloads.config_inputs(name, rows=min(c["rows"], 8))
    idx0, val0 = oracle.topk(bits, c["dtype"], c["k"], row_len=row_len)
    for seed in [0x5EED5EED, 1, 2]:
        idx, val, stats = oracle.model(bits, c["dtype"], c["k"], c["B"], c["B2"], seed,
                                       row_len=row_len)
        np.testing.assert_array_equal(idx, idx0)
        np.testing.assert_array_equal(val, val0)
        check_identities(stats, c["k"], c["B"], c["B2"])


@pytest.mark.parametrize("splits", [2, 3, 8, 16])
def test_model_split_rows_match_definition(splits):
    bits, row_len = workloads.generate(6, 20000, "fp32", "ragged_normal", seed=31, min_len=1)
    row_len[0] = 5          # fewer blocks than slices
    k, B, B2 = 300, 256, 512
    idx0, val0 = oracle.topk(bits, "fp32", k, row_len=row_len)
    idx, val, stats = oracle.model(bits, "fp32", k, B, B2, 77, row_len=row_len, splits=splits)
    np.testing.assert_array_equal(idx, idx0)
    np.testing.assert_array_equal(val, val0)
    check_identities(stats, k, B, B2)
    assert stats.shape == (6, splits, 4)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("kind", ["levels", "specials", "constant", "ascending"])
def test_model_matches_definition_with_ties_and_specials(dtype, kind):
    bits, _ = workloads.generate(4, 9000, dtype, kind, seed=41)
    for k, B, B2 in [(1, 1, 1), (64, 100, 37), (500, 128, 128), (9000, 512, 64)]:
        idx0, val0 = oracle.topk(bits, dtype, k)
        idx, val, stats = oracle.model(bits, dtype, k, B, B2, 123)
        np.testing.assert_array_equal(idx, idx0)
        np.testing.assert_array_equal(val, val0)
        check_identities(stats, k, B, B2)


def test_model_rows_shorter_than_k():
    bits, _ = workloads.generate(3, 100, "fp32", "normal", seed=2)
    row_len = np.array([0, 7, 100], dtype=np.int32)
    idx0, val0 = oracle.topk(bits, "fp32", 50, row_len=row_len)
    idx, val, stats = oracle.model(bits, "fp32", 50, 8, 8, 9, row_len=row_len)
    np.testing.assert_array_equal(idx, idx0)
    np.testing.assert_array_equal(val, val0)
    assert stats[0, 0].tolist() == [0, 0, 0, 0]
    assert stats[1, 0].tolist() == [7, 0, 7, 7]


@pytest.mark.parametrize("case", [
    dict(kind="normal", N=4096, k=64, B=128, B2=128),
    dict(kind="ascending", N=65536, k=256, B=256, B2=256),
    dict(kind="levels", N=65536, k=512, B=512, B2=512),
    dict(kind="normal", N=32768, k=512, B=1024, B2=1024),
])
def test_expected_work_bound(case):
    """Mean W over 200 random block orders stays under the page's bound."""
    bits, _ = workloads.generate(1, case["N"], "fp32", case["kind"], seed=55)
    Ws = []
    for seed in range(200):
        _, _, stats = oracle.model(bits, "fp32", case["k"], case["B"], case["B2"], 1000 + seed)
        check_identities(stats, case["k"], case["B"], case["B2"])
        Ws.append(int(stats[0, 0, 2]))
    Ws = np.array(Ws, dtype=np.float64)
    bound = w_bound(case["N"], case["k"], case["B"], case["B2"])
    mean, sem = Ws.mean(), Ws.std(ddof=1) / math.sqrt(len(Ws))
    assert mean + 3 * sem <= bound, (mean, sem, bound)


def test_identity_order_blows_up_on_ascending_rows():
    """Without the random order an ascending row appends every element: the
    reason the page requires a random block order."""
    N, k, B, B2 = 65536, 256, 256, 256
    bits, _ = workloads.generate(1, N, "fp32", "ascending", seed=56)
    _, _, st = oracle.model(bits, "fp32", k, B, B2, 0, identity_order=True)
    A, R, W, _ = st[0, 0]
    assert A == N
    assert W > 5 * w_bound(N, k, B, B2)
    _, _, st_random = oracle.model(bits, "fp32", k, B, B2, 0)
    assert st_random[0, 0, 2] < w_bound(N, k, B, B2)
