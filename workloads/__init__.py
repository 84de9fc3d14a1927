"""Seeded synthetic inputs for DeepSelect top-k.

This module only draws input data: it holds none of the top-k arithmetic and
is shared by the tests, the benchmark and the CPU oracle's callers alike.
Values are drawn in float32 with numpy's PCG64 generator (platform
independent) and, for bf16 workloads, rounded to bfloat16 by torch's
round-to-nearest-even conversion.  Arrays come back as raw bit patterns
(uint32 for fp32, uint16 for bf16) so that every consumer sees exactly the
same bytes.

The five named workloads stand in for the two uses the DeepSelect page names
(PFCCLab/DeepSelect "DeepSelect-deep-dive", section "算法设计背景": choosing
context tokens in DeepSeek Sparse Attention and candidate tokens during
sampling) plus a small case and an adversarial case; no real scores or logits
are used.
"""
import numpy as np

FP32 = "fp32"
BF16 = "bf16"
FP16 = "fp16"

# name -> shape, dtype, selection parameters, value recipe and data seed
CONFIGS = {
    "small_fp32": dict(rows=1, N=4096, dtype=FP32, k=64, B=128, B2=128,
                       kind="normal", seed=1001,
                       desc="1 x 4096 fp32 N(0,1), k=64, B=B2=128"),
    "dsa_index_bf16": dict(rows=64, N=32768, dtype=BF16, k=512, B=1024, B2=1024,
                           kind="normal", seed=1002,
                           desc="DSA index scores: 64 x 32768 bf16 N(0,1), k=512, B=B2=1024"),
    "dsa_decode_ragged_fp32": dict(rows=8, N=131072, dtype=FP32, k=2048, B=2048, B2=2048,
                                   kind="ragged_normal", seed=1003,
                                   desc="DSA long-context decode: 8 x 131072 fp32 N(0,1), "
                                        "row_len uniform in [2048, N], +inf past row_len, "
                                        "k=2048, B=B2=2048"),
    "sampling_logits_bf16": dict(rows=256, N=128000, dtype=BF16, k=50, B=1024, B2=1024,
                                 kind="gumbel_spikes", seed=1004,
                                 desc="sampling logits: 256 x 128000 bf16 Gumbel(0,1) "
                                      "+8 at 32 distinct columns per row, k=50, B=B2=1024"),
    "adversarial_fp32": dict(rows=32, N=262144, dtype=FP32, k=1024, B=1024, B2=1024,
                             kind="adversarial", seed=1005,
                             desc="adversarial: 32 x 262144 fp32, rows 0-15 sorted ascending "
                                  "N(0,1), rows 16-31 from 16 levels, k=1024, B=B2=1024"),
}

CONFIG_ORDER = ["small_fp32", "dsa_index_bf16", "dsa_decode_ragged_fp32",
                "sampling_logits_bf16", "adversarial_fp32"]

# one row over the whole GPU (ds_topk_long_row): the single huge row of the
# multi-pass selection in "CUDA 算子笔记 4", section "Top K Selection"
LONG_ROW = dict(rows=1, N=1 << 27, dtype=FP32, k=1024, B=1024, B2=1024, kind="normal", seed=1006,
                desc="one long row: 1 x 2^27 fp32 N(0,1), k=1024, B=B2=1024")


def to_bf16_bits(f32):
    """Round float32 values to bfloat16 (nearest even) and return the uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def to_f16_bits(f32):
    """IEEE binary16 bit patterns of float32 values (round to nearest even)."""
    return np.ascontiguousarray(np.asarray(f32, dtype=np.float32).astype(np.float16)).view(np.uint16)


def bits_to_f32(bits, dtype):
    """Widen bit patterns to float32 values (exact for bf16 and fp16)."""
    if dtype == FP32:
        return np.asarray(bits, dtype=np.uint32).view(np.float32)
    if dtype == FP16:
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _finish(f32, dtype):
    if dtype == FP32:
        return np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    if dtype == FP16:
        return to_f16_bits(f32)
    return to_bf16_bits(f32)


def generate(rows, N, dtype, kind, seed, **kw):
    """Draw a [rows, N] input.  Returns (bits, row_len or None).

    kinds:
      normal         i.i.d. N(0,1)
      ragged_normal  N(0,1); row_len[r] uniform in [min_len, N] (inclusive);
                     columns at or past row_len hold +inf (must never be read)
      gumbel_spikes  -log(-log(U)), U uniform in (0,1), plus +spike at
                     `spikes` distinct random columns of each row
      adversarial    first half of the rows: sorted ascending N(0,1);
                     second half: integers drawn from `levels` levels 0..levels-1
      ascending      sorted ascending N(0,1) in every row
      levels         integers 0..levels-1
      constant       every element equal to `value`
      specials       N(0,1) mixed with NaN, +-0, +-inf, denormals and repeats
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    row_len = None
    if kind == "normal":
        f = rng.standard_normal((rows, N), dtype=np.float32)
    elif kind == "ragged_normal":
        f = rng.standard_normal((rows, N), dtype=np.float32)
        lo = int(kw.get("min_len", min(2048, N)))
        row_len = rng.integers(lo, N + 1, size=rows, dtype=np.int64).astype(np.int32)
        cols = np.arange(N)[None, :]
        f[cols >= row_len[:, None]] = np.inf
    elif kind == "gumbel_spikes":
        u = rng.random((rows, N), dtype=np.float64)
        u = np.where(u == 0.0, np.nextafter(0.0, 1.0), u)   # open interval (0, 1)
        f = (-np.log(-np.log(u))).astype(np.float32)
        spikes = int(kw.get("spikes", 32))
        spike = float(kw.get("spike", 8.0))
        for r in range(rows):
            cols = rng.permutation(N)[:spikes]
            f[r, cols] += np.float32(spike)
    elif kind == "adversarial":
        half = rows // 2
        levels = int(kw.get("levels", 16))
        f = np.empty((rows, N), dtype=np.float32)
        f[:half] = np.sort(rng.standard_normal((half, N), dtype=np.float32), axis=1)
        f[half:] = rng.integers(0, levels, size=(rows - half, N)).astype(np.float32)
    elif kind == "ascending":
        f = np.sort(rng.standard_normal((rows, N), dtype=np.float32), axis=1)
    elif kind == "levels":
        levels = int(kw.get("levels", 16))
        f = rng.integers(0, levels, size=(rows, N)).astype(np.float32)
    elif kind == "constant":
        f = np.full((rows, N), np.float32(kw.get("value", 1.0)), dtype=np.float32)
    elif kind == "specials":
        f = rng.standard_normal((rows, N), dtype=np.float32)
        pool = np.array([np.nan, -np.nan, 0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-40,
                         3.0, 3.0, -2.5], dtype=np.float32)
        pick = rng.random((rows, N)) < float(kw.get("fraction", 0.05))
        f[pick] = pool[rng.integers(0, len(pool), size=int(pick.sum()))]
        bits = f.view(np.uint32)
        nan_mask = np.isnan(f)
        # distinct NaN payloads, both signs: the oracle must return the bits as read
        payload = rng.integers(1, 1 << 22, size=int(nan_mask.sum()), dtype=np.uint32)
        bits[nan_mask] = (bits[nan_mask] & np.uint32(0xFFC00000)) | payload
    else:
        raise ValueError("unknown kind %r" % kind)
    out = _finish(f, dtype)
    if kind == "specials" and dtype == FP16:
        # the narrowing canonicalises NaNs: give them distinct 10-bit payloads
        nan16 = (out & np.uint16(0x7C00)) == np.uint16(0x7C00)
        nan16 &= (out & np.uint16(0x03FF)) != 0
        pl = rng.integers(1, 1 << 10, size=int(nan16.sum()), dtype=np.uint32).astype(np.uint16)
        out[nan16] = (out[nan16] & np.uint16(0xFC00)) | pl
    return out, row_len


def config_inputs(name, rows=None):
    """Input of a named workload; `rows` optionally keeps only the first rows."""
    c = CONFIGS[name]
    bits, row_len = generate(c["rows"], c["N"], c["dtype"], c["kind"], c["seed"])
    if rows is not None:
        bits = bits[:rows]
        row_len = None if row_len is None else row_len[:rows]
    return bits, row_len


def algorithmic_bytes(name_or_cfg, row_len=None, rows=None):
    """Bytes the method must move: every valid input element read once, the
    k outputs written (int32 index + value), and row_len read when given."""
    c = CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    s = 4 if c["dtype"] == FP32 else 2
    n_rows = c["rows"] if rows is None else rows
    if row_len is None:
        read = n_rows * c["N"] * s
        meta = 0
    else:
        read = int(np.clip(np.asarray(row_len, dtype=np.int64), 0, c["N"]).sum()) * s
        meta = 4 * n_rows
    return read + n_rows * c["k"] * (4 + s) + meta
