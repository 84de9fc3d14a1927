"""Pins for the oracle's Philox4x32-10 and the block permutation (CPU only).

Philox4x32-10 is defined in Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3" (SC'11).  The oracle's implementation is checked
against (a) the known-answer vectors distributed with that paper's reference
library (Random123, file kat_vectors, "philox4x32 10" lines), and (b) cuRAND's
host-side PHILOX4_32_10 generator, a library routine that runs on the CPU:
for seed s and generator offset 4*i its first four words are Philox4x32-10 of
counter (i div 2^16, 0, i mod 2^16, 0) under key (s mod 2^32, s div 2^32).
"""
import ctypes
import ctypes.util

import numpy as np
import pytest

import oracle

KAT = [
    # counter (4 words), key (2 words), output (4 words)
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff, 0xffffffff, 0xffffffff, 0xffffffff), (0xffffffff, 0xffffffff),
     (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
]


@pytest.mark.parametrize("ctr,key,out", KAT)
def test_philox_known_answers(ctr, key, out):
    assert oracle.philox(ctr, key).tolist() == list(out)


def _curand():
    for name in ["libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand")]:
        for prefix in ["/usr/local/cuda/lib64/", ""]:
            if not name:
                continue
            try:
                return ctypes.CDLL(prefix + name)
            except OSError:
                continue
    return None


def test_philox_matches_curand_host_generator():
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    PHILOX4_32_10 = 161
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), PHILOX4_32_10) != 0:
        pytest.skip("cuRAND host generator unavailable")
    try:
        rng = np.random.default_rng(0)
        seeds = [0, 1, 0xFFFFFFFF, 0x100000000, 0x5EED5EED, 0x0123456789ABCDEF] + \
            [int(s) for s in rng.integers(0, 1 << 63, size=20)]
        for seed in seeds:
            for i in [0, 1, 2, 77, 65535, 65536, 123456, 0xFFFFFFF]:
                assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
                assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * i)) == 0
                buf = (ctypes.c_uint * 4)()
                assert lib.curandGenerate(gen, buf, 4) == 0
                mine = oracle.philox((i >> 16, 0, i & 0xFFFF, 0), (seed & 0xFFFFFFFF, seed >> 32))
                assert mine.tolist() == list(buf), (hex(seed), i)
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("m,first", [(1, 0), (7, 0), (125, 0), (256, 0), (64, 192)])
def test_permutation_is_a_permutation(m, first):
    for seed in [0, 1, 0x5EED5EED]:
        for row, sl in [(0, 0), (3, 1), (255, 7)]:
            p = oracle.permutation(m, seed, row, sl, first)
            assert sorted(p.tolist()) == list(range(first, first + m))


def test_permutation_follows_philox_word_order():
    m, seed, row, sl, first = 40, 0xABCDEF0123, 5, 2, 80
    words = [int(oracle.philox((first + i, row, sl, 0), (seed & 0xFFFFFFFF, seed >> 32))[0])
             for i in range(m)]
    expected = [first + i for _, i in sorted((w, i) for i, w in enumerate(words))]
    assert oracle.permutation(m, seed, row, sl, first).tolist() == expected


def test_permutation_positions_are_uniform():
    """Chi-square: each block lands in each position equally often."""
    m, trials = 8, 4000
    counts = np.zeros((m, m))
    for s in range(trials):
        p = oracle.permutation(m, 10_000 + s, 0, 0, 0)
        counts[np.arange(m), p] += 1
    expected = trials / m
    chi2 = ((counts - expected) ** 2 / expected).sum(axis=1)
    # 7 degrees of freedom per row; 0.1% critical value is 24.32
    assert chi2.max() < 24.32 * 1.2, chi2


def test_permutation_depends_on_seed_row_and_slice():
    base = oracle.permutation(64, 1, 0, 0, 0).tolist()
    assert oracle.permutation(64, 2, 0, 0, 0).tolist() != base
    assert oracle.permutation(64, 1, 1, 0, 0).tolist() != base
    assert oracle.permutation(64, 1, 0, 1, 0).tolist() != base
