"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign or index, a transposed operand), compiles the copy into a
temporary library and runs a battery of the pins from the other oracle test
files against it, in a child process (a mutant that reads out of bounds may
crash, which counts as caught).  Every mutant must fail at least one pin; the
unmodified source must pass all of them.
"""
import json
import math
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import oracle
import workloads

SRC = os.path.join(os.path.dirname(oracle.__file__), "ds_oracle.c")

MUTANTS = {
    "tie_break_reversed": ("    return a.idx < b.idx;\n}", "    return a.idx > b.idx;\n}"),
    "negative_zero_not_merged": ("    if (magnitude == 0u)              /* -0.0 and +0.0 */\n"
                                 "        return 0x80000000u;\n", ""),
    "nan_not_canonical": ("    if (magnitude > 0x7F800000u)      /* NaN, any sign or payload */\n"
                          "        return 0xFFFFFFFFu;\n", ""),
    "negative_not_flipped": ("        return ~bits;\n", "        return bits;\n"),
    "bf16_sign_bit_wrong": ("        return 0xFFFFu;\n    if (magnitude == 0u)\n        return 0x8000u;\n    if (bits & 0x8000u)\n        return (~bits) & 0xFFFFu;\n    return bits | 0x8000u;\n}\n\n/* IEEE",
                            "        return 0xFFFFu;\n    if (magnitude == 0u)\n        return 0x8000u;\n    if (bits & 0x8000u)\n        return (~bits) & 0xFFFFu;\n    return bits | 0x4000u;\n}\n\n/* IEEE"),
    "fp16_inf_taken_as_nan": ("    if (magnitude > 0x7C00u)\n", "    if (magnitude >= 0x7C00u)\n"),
    "row_len_not_clamped": ("    if (len > N)\n        len = N;\n", ""),
    "threshold_is_largest": ("threshold = cand[n - 1];", "threshold = cand[0];"),
    "filter_operands_swapped": ("pair_before(p, threshold)", "pair_before(threshold, p)"),
    "trigger_strict": ("if (n >= (int64_t)k + B2) {", "if (n > (int64_t)k + B2) {"),
    "final_call_not_counted": ("            W += n;                            /* the final TopK call */\n",
                               ""),
    "philox_multipliers_swapped": ("uint64_t p0 = (uint64_t)M0 * c0;", "uint64_t p0 = (uint64_t)M1 * c0;"),
    "philox_key_bumped_early": ("        if (round > 0) {", "        if (round >= 0) {"),
    "philox_words_crossed": ("uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;",
                             "uint32_t n0 = (uint32_t)(p0 >> 32) ^ c1 ^ k0;"),
    "permutation_descending": ("        return a.word < b.word ? -1 : 1;", "        return a.word > b.word ? -1 : 1;"),
    "slices_overlap": ("int64_t first = (int64_t)c * per_slice;", "int64_t first = (int64_t)c * per_slice / 2;"),
}

KAT0 = ((0, 0, 0, 0), (0, 0), [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8])
KAT1 = ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
        [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1])
SPECIALS = [-math.inf, -1.0, -0.0, 0.0, 1.0, 2.0, math.inf, math.nan, -math.nan]


def _brute_order(f):
    rows, n = f.shape
    a, b = f[:, :, None], f[:, None, :]
    na, nb = np.isnan(a), np.isnan(b)
    with np.errstate(invalid="ignore"):
        before = (na & ~nb) | ((a > b) & ~na & ~nb) | \
            ((((a == b) & ~na & ~nb) | (na & nb)) & (np.arange(n)[None, :, None] < np.arange(n)[None, None, :]))
    return np.argsort(before.sum(axis=1), axis=1)


def _battery(lib):
    """Names of the pins that fail for this oracle library."""
    failed = []

    def check(name, fn):
        try:
            if not fn():
                failed.append(name)
        except Exception:      # a crash or a rejected call is a failure too
            failed.append(name)

    x = np.array([[1, 5, 3, 2, 4]], dtype=np.float32)
    check("worked_example", lambda: oracle.topk(x, "fp32", 3, lib=lib)[0].tolist() == [[1, 4, 2]])

    import itertools
    combos = np.array(list(itertools.product(range(len(SPECIALS)), repeat=4)))
    f = np.array(SPECIALS, dtype=np.float32)[combos]
    order = _brute_order(f)
    for dt in ["fp32", "bf16", "fp16"]:
        bits = f.view(np.uint32) if dt == "fp32" else \
            workloads.to_bf16_bits(f) if dt == "bf16" else workloads.to_f16_bits(f)
        check("brute_force_" + dt,
              lambda b=bits, d=dt: np.array_equal(oracle.topk(b, d, 2, lib=lib)[0], order[:, :2]))

    sp_bits, _ = workloads.generate(64, 300, "fp32", "specials", seed=4, fraction=0.05)
    check("argmax_specials", lambda: np.array_equal(
        oracle.topk(sp_bits, "fp32", 1, lib=lib)[0][:, 0], np.argmax(sp_bits.view(np.float32), axis=1)))

    rl_bits, _ = workloads.generate(2, 64, "fp32", "normal", seed=12)
    check("row_len_clamp", lambda: np.array_equal(
        oracle.topk(rl_bits, "fp32", 10, row_len=np.array([1000, 64], np.int32), lib=lib)[0],
        oracle.topk(rl_bits, "fp32", 10, lib=lib)[0]))

    check("philox_kat0", lambda: oracle.philox(*KAT0[:2], lib=lib).tolist() == KAT0[2])
    check("philox_kat1", lambda: oracle.philox(*KAT1[:2], lib=lib).tolist() == KAT1[2])

    def perm_order():
        m, seed = 30, 99
        w = [int(oracle.philox((i, 0, 0, 0), (seed, 0), lib=lib)[0]) for i in range(m)]
        return oracle.permutation(m, seed, 0, 0, 0, lib=lib).tolist() == \
            [i for _, i in sorted((w[i], i) for i in range(m))]
    check("permutation_order", perm_order)

    def model_cases():
        ok = True
        for kind, N, k, B, B2, splits in [("normal", 3000, 64, 128, 128, 1),
                                          ("levels", 3000, 300, 64, 64, 1),
                                          ("specials", 2000, 1, 1, 1, 1),
                                          ("normal", 5000, 100, 64, 256, 4)]:
            bits, _ = workloads.generate(2, N, "fp32", kind, seed=3)
            ref = oracle.topk(bits, "fp32", k, lib=lib)
            idx, val, st = oracle.model(bits, "fp32", k, B, B2, 5, splits=splits, lib=lib)
            A, R, W, peak = st[..., 0], st[..., 1], st[..., 2], st[..., 3]
            ok &= np.array_equal(idx, ref[0]) and np.array_equal(val, ref[1])
            ok &= bool(np.all(W == A + k * R)) and bool(np.all(R * B2 <= A))
            ok &= bool(np.all(peak <= k + B2 + B - 1))
            ok &= bool(np.all(A <= -(-N // splits) + B))
        return ok
    check("model_identities", model_cases)
    return failed


def _compile(source_text, tmpdir, name):
    src = os.path.join(tmpdir, name + ".c")
    with open(src, "w") as f:
        f.write(source_text)
    out = os.path.join(tmpdir, name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", out, src], check=True)
    return out


def _battery_in_child(lib_path):
    """Run the battery in a fresh interpreter; None means the child crashed."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), lib_path],
                          capture_output=True, text=True, env=env, timeout=600)
    if proc.returncode != 0:
        return None
    return json.loads(proc.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def original_source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_oracle_passes_battery(original_source, tmp_path):
    path = _compile(original_source, str(tmp_path), "original")
    assert _battery_in_child(path) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, original_source):
    old, new = MUTANTS[name]
    assert original_source.count(old) == 1, "mutation site not found: " + name
    with tempfile.TemporaryDirectory() as d:
        path = _compile(original_source.replace(old, new), d, name)
        failed = _battery_in_child(path)
        assert failed is None or failed, "mutant %s passed every pin" % name


if __name__ == "__main__":
    print(json.dumps(_battery(oracle.load(sys.argv[1]))))
