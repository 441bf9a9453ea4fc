"""Seeded synthetic inputs for the fused FP8 MQA-logits + top-k prefill path.

This module only *makes inputs*: it draws numbers, rounds them to the FP8 e4m3fn
storage format the op consumes, and lays out row ranges.  It holds none of the
scoring or selection arithmetic, so both the CPU oracle and the CUDA path can
take their inputs from here without sharing any of the method's code.

Input contract (vLLM API page `vllm.model_executor.kernels.attention.dsa.
fused_mqa_topk`, `fused_mqa_topk_prefill` docstring): q is [rows, 32, 128] fp8
e4m3, k is [keys, 128] fp8 e4m3, weights [rows, 32] fp32, starts/ends [rows]
int32, top-k in {512, 1024, 2048}.  Key scales arrive as the indexer cache's
[keys, 4] uint8 UE8M0 bytes (four equal exponent bytes per key,
`fused_mqa_topk_key_scales` docstring).

Recipe (shared by every config): q and k are N(0,1) fp32 rounded to e4m3fn
(round-to-nearest-even, saturating at +-448); weights are N(0,1)/sqrt(32);
UE8M0 exponents are uniform integers in [120, 127].  One numpy
``default_rng(seed)`` per config with a fixed draw order: q, k, weights, scale
exponents, then the variant draws.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEADS = 32
HEAD_DIM = 128
TOPKS = (512, 1024, 2048)

E4M3_MAX = 448.0


def quantize_e4m3fn(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to e4m3fn storage codes (uint8), RNE, saturating.

    e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
    0x7F/0xFF are NaN, so the largest finite magnitude is 1.75 * 2**8 = 448.
    Subnormals are m * 2**-9 for m in 1..7.
    """
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("quantize_e4m3fn: non-finite input")
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.minimum(np.abs(x).astype(np.float64), E4M3_MAX)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: value = m * 2^-9; rint is round-half-even; m == 8 is the
    # smallest normal (code 0x08), which the encoding reaches continuously.
    code[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    if np.any(nrm):
        an = a[nrm]
        e = np.floor(np.log2(an)).astype(np.int64)
        # guard log2 rounding at exact powers of two
        e = np.where(np.ldexp(1.0, e) > an, e - 1, e)
        e = np.where(np.ldexp(1.0, e + 1) <= an, e + 1, e)
        m = np.rint(np.ldexp(an, -e) * 8.0 - 8.0).astype(np.int64)  # 0..8
        carry = m == 8
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 0, m)
        c = ((e + 7) << 3) | m
        c = np.minimum(c, 0x7E)  # saturate (448 is 0x7E)
        code[nrm] = c
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def quantize_e4m3fn_fast(x: np.ndarray) -> np.ndarray:
    """Same codes as `quantize_e4m3fn` for large arrays: saturate to +-448,
    then torch's round-to-nearest-even float8_e4m3fn cast (chunked)."""
    import torch
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    xf, of = x.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for i in range(0, xf.size, step):
        t = torch.from_numpy(xf[i:i + step]).clamp(-E4M3_MAX, E4M3_MAX)
        of[i:i + step] = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out


def ue8m0_bytes(exponents: np.ndarray) -> np.ndarray:
    """Pack per-key exponents as the cache's [keys, 4] uint8 groups (4 equal bytes)."""
    e = np.asarray(exponents, dtype=np.uint8)
    return np.repeat(e[:, None], 4, axis=1).copy()


@dataclasses.dataclass
class Problem:
    """One prefill chunk: raw input bytes plus its row ranges."""
    name: str
    q: np.ndarray          # uint8 [rows, 32, 128] e4m3fn codes
    k: np.ndarray          # uint8 [keys, 128] e4m3fn codes
    scales_ue8m0: np.ndarray  # uint8 [keys, 4]
    weights: np.ndarray    # float32 [rows, 32]
    starts: np.ndarray     # int32 [rows]
    ends: np.ndarray       # int32 [rows]
    topk: int
    # rows whose weights were scaled (adversarial variant), for sampling
    special_rows: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def keys(self) -> int:
        return int(self.k.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def dim(self) -> int:
        return int(self.q.shape[2])

    def visible(self) -> np.ndarray:
        return np.maximum(self.ends.astype(np.int64) - self.starts.astype(np.int64), 0)

    def pairs(self) -> int:
        return int(self.visible().sum())


def _draw_core(rng, rows, keys, heads=HEADS, dim=HEAD_DIM, k_offset_dim0: float = 0.0):
    qf = rng.standard_normal((rows, heads, dim), dtype=np.float32)
    kf = rng.standard_normal((keys, dim), dtype=np.float32)
    if k_offset_dim0:
        kf[:, 0] += np.float32(k_offset_dim0)
    w = (rng.standard_normal((rows, heads), dtype=np.float32) / np.float32(math.sqrt(heads))).astype(np.float32)
    exps = rng.integers(120, 128, size=keys, dtype=np.int64).astype(np.uint8)
    quant = quantize_e4m3fn if qf.size + kf.size <= (1 << 22) else quantize_e4m3fn_fast
    return quant(qf), quant(kf), w, exps


def causal_tail(rows: int, keys: int, base: int = 0):
    """Rows are the last `rows` tokens of a `keys`-token context: row i sees
    [base, base + keys - rows + i + 1)."""
    i = np.arange(rows, dtype=np.int64)
    starts = np.full(rows, base, dtype=np.int64)
    ends = base + keys - rows + i + 1
    return starts.astype(np.int32), ends.astype(np.int32)


def make_single(name, rows, keys, topk, seed=0, k_offset_dim0=0.0,
                dup_frac=0.0, scaled_row_frac=0.0, scaled_row_factor=1e6,
                heads=HEADS, dim=HEAD_DIM) -> Problem:
    """Single-request chunk with a causal tail (every config but the 4-request one)."""
    rng = np.random.default_rng(seed)
    q, k, w, exps = _draw_core(rng, rows, keys, heads, dim, k_offset_dim0)
    special = np.zeros(0, np.int64)
    if dup_frac > 0:
        nd = int(round(keys * dup_frac))
        dst = rng.choice(keys, size=nd, replace=False)
        src = rng.integers(0, keys, size=nd)
        k[dst] = k[src]
        exps[dst] = exps[src]
    if scaled_row_frac > 0:
        ns = max(1, int(round(rows * scaled_row_frac)))
        special = np.sort(rng.choice(rows, size=ns, replace=False))
        w[special] = (w[special] * np.float32(scaled_row_factor)).astype(np.float32)
    starts, ends = causal_tail(rows, keys)
    return Problem(name, q, k, ue8m0_bytes(exps), w, starts, ends, topk, special)


def make_multi(name, contexts, row_split, topk, seed=0) -> Problem:
    """Multi-request chunk: K is the concatenation of each request's keys; a
    request with context N_q and R_q rows contributes rows whose range is
    [b_q, b_q + N_q - R_q + t + 1) for t < R_q (causal within the request)."""
    rows = int(sum(row_split))
    keys = int(sum(contexts))
    rng = np.random.default_rng(seed)
    q, k, w, exps = _draw_core(rng, rows, keys)
    starts = np.empty(rows, np.int32)
    ends = np.empty(rows, np.int32)
    r0, base = 0, 0
    for n_q, r_q in zip(contexts, row_split):
        s, e = causal_tail(r_q, n_q, base)
        starts[r0:r0 + r_q] = s
        ends[r0:r0 + r_q] = e
        r0 += r_q
        base += n_q
    return Problem(name, q, k, ue8m0_bytes(exps), w, starts, ends, topk)


# The chunk shapes of the workload table: 16,384-row prefill chunks at top-2048
# with 32K..1M keys, multi-request chunks, the 512/1024/2048 top-k set; and
# decode batches of few rows per request.
CONFIGS = {
    "tiny_64x4096_k512": lambda: make_single("tiny_64x4096_k512", 64, 4096, 512),
    "r2048_32k_k512": lambda: make_single("r2048_32k_k512", 2048, 32768, 512),
    "r2048_32k_k2048": lambda: make_single("r2048_32k_k2048", 2048, 32768, 2048),
    "r16k_128k_k2048": lambda: make_single("r16k_128k_k2048", 16384, 131072, 2048),
    "r16k_128k_k2048_offset4": lambda: make_single("r16k_128k_k2048_offset4", 16384, 131072, 2048,
                                                   k_offset_dim0=4.0),
    "multi4_r16k_k1024": lambda: make_multi("multi4_r16k_k1024", (300, 4096, 65536, 262144),
                                            (64, 1024, 5312, 9984), 1024),
    "r16k_1m_k2048": lambda: make_single("r16k_1m_k2048", 16384, 1 << 20, 2048),
    "r16k_1m_k2048_adversarial": lambda: make_single("r16k_1m_k2048_adversarial", 16384, 1 << 20, 2048,
                                                     dup_frac=0.25, scaled_row_frac=0.01),
    # 64 index heads per query row (DeepSeek-V3.2's indexer), prefill chunk
    "h64_r2048_64k_k2048": lambda: make_single("h64_r2048_64k_k2048", 2048, 65536, 2048, heads=64),
    # Decode batches: each request verifies K + 1 = 8 query rows (speculative
    # K = 7) against its own context; row t of a request sees its context up to
    # N - 8 + t + 1 keys (the multi-request layout with 8 rows per request).
    "decode_b32_s8_64k_k2048": lambda: make_multi("decode_b32_s8_64k_k2048", (65536,) * 32, (8,) * 32, 2048),
    "decode_b4_s8_256k_k2048": lambda: make_multi("decode_b4_s8_256k_k2048", (262144,) * 4, (8,) * 4, 2048),
    "decode_b64_s8_mixed_k512": lambda: make_multi(
        "decode_b64_s8_mixed_k512", tuple((4096, 8192, 16384, 32768, 65536, 131072)[i % 6] for i in range(64)),
        (8,) * 64, 512),
}


def make(name: str) -> Problem:
    return CONFIGS[name]()


def random_small(seed: int, rows: int, keys: int, topk: int, heads=HEADS, dim=HEAD_DIM,
                 empty_frac: float = 0.1) -> Problem:
    """Small randomised chunk with arbitrary [start, end) ranges (some empty,
    some shorter than top-k, some reversed) for parity sweeps."""
    rng = np.random.default_rng(seed)
    q, k, w, exps = _draw_core(rng, rows, keys, heads, dim)
    a = rng.integers(0, keys + 1, size=rows)
    b = rng.integers(0, keys + 1, size=rows)
    starts = np.minimum(a, b)
    ends = np.maximum(a, b)
    emp = rng.random(rows) < empty_frac
    ends[emp] = starts[emp]  # empty rows
    return Problem(f"random_{seed}", q, k, ue8m0_bytes(exps), w, starts.astype(np.int32),
                   ends.astype(np.int32), topk)


MAX_KEYS = 1 << 24  # the largest key count the library accepts


def max_keys(seed: int = 90, rows: int = 16, used: int = 400_000, topk: int = 2048) -> Problem:
    """A chunk at the largest key count (2^24 keys: K is 2 GiB).  Row 0 sees
    the last `used` keys (long enough to be gated), row 1 the first 5000,
    rows 2-4 end at the last key with 1, k - 1 and k + 1 keys, and the rest
    have random ranges inside the last `used` keys.  Only keys that some row
    sees are drawn; the others hold code 0."""
    rng = np.random.default_rng(seed)
    keys, lo, head = MAX_KEYS, MAX_KEYS - used, 8192
    q = quantize_e4m3fn_fast(rng.standard_normal((rows, HEADS, HEAD_DIM), dtype=np.float32))
    w = (rng.standard_normal((rows, HEADS), dtype=np.float32) / np.float32(math.sqrt(HEADS))).astype(np.float32)
    k = np.zeros((keys, HEAD_DIM), np.uint8)
    k[lo:] = quantize_e4m3fn_fast(rng.standard_normal((used, HEAD_DIM), dtype=np.float32))
    k[:head] = quantize_e4m3fn_fast(rng.standard_normal((head, HEAD_DIM), dtype=np.float32))
    exps = np.full(keys, 127, np.uint8)
    exps[lo:] = rng.integers(120, 128, size=used).astype(np.uint8)
    exps[:head] = rng.integers(120, 128, size=head).astype(np.uint8)
    starts = np.empty(rows, np.int64)
    ends = np.empty(rows, np.int64)
    fixed = [(lo, keys), (0, 5000), (keys - 1, keys), (keys - (topk - 1), keys), (keys - (topk + 1), keys)]
    for i in range(rows):
        if i < len(fixed):
            starts[i], ends[i] = fixed[i]
        else:
            a, b = np.sort(rng.integers(lo, keys + 1, size=2))
            starts[i], ends[i] = a, b
    return Problem(f"max_keys_{seed}", q, k, ue8m0_bytes(exps), w, starts.astype(np.int32), ends.astype(np.int32),
                   topk)


def window(p: Problem, r: int) -> Problem:
    """Row r of p alone, with K cut to the row's range (indices relative to
    the range start are unchanged)."""
    s, e = int(p.starts[r]), int(p.ends[r])
    return Problem(f"{p.name}_row{r}", p.q[r:r + 1], p.k[s:e], p.scales_ue8m0[s:e], p.weights[r:r + 1],
                   np.zeros(1, np.int32), np.array([e - s], np.int32), p.topk)


def sample_rows(p: Problem, count: int, seed: int = 1234) -> np.ndarray:
    """Deterministic row sample for checks and CPU timing on big chunks: evenly
    spaced rows, the first and last row, every specially treated row (capped),
    and every row that sees fewer than top-k keys."""
    rows = p.rows
    picks = set(np.linspace(0, rows - 1, num=max(2, count), dtype=np.int64).tolist())
    picks.update([0, rows - 1])
    if p.special_rows.size:
        picks.update(p.special_rows[: max(4, count // 4)].tolist())
    short = np.nonzero(p.visible() < p.topk)[0]
    picks.update(short[:256].tolist())
    return np.array(sorted(picks), dtype=np.int64)


def small_subproblem(p: Problem, rows: np.ndarray) -> Problem:
    """The same keys with only the chosen rows (used to time the oracle on a sample)."""
    rows = np.asarray(rows, dtype=np.int64)
    return Problem(p.name + "_sample", p.q[rows], p.k, p.scales_ue8m0, p.weights[rows],
                   p.starts[rows], p.ends[rows], p.topk)
