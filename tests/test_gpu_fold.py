"""Parity of the fold compilation of the fused kernel (head_sum = 1): the
weighted linear half of relu(s) = (s + |s|) / 2 runs on the tensor core as the
row's folded query in four e4m3 terms (vLLM pull request #60618, "What this PR
does", Scoring bullet), and a row whose fold error bound is too large for its
scores ("weights unsafe to scale", same section, Exact rescan bullet) is
rescanned exactly with the direct head sum.  Every case is checked against the
oracle under the pass rule of the other parity tests."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_topk_rows, to_device

pytestmark = pytest.mark.gpu

FOLD = {"head_sum": 1}


@pytest.fixture(scope="module")
def mqa():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_attention_indexer_relu_gb300 as m
    m.lib()
    return m


def run(mqa, p, debug):
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows)
    out = mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk, workspace=ws, debug=debug)
    status, stats = mqa.get_status(ws)
    return out.cpu().numpy(), status, stats


def assert_parity(p, got, rows=None):
    rows = np.arange(p.rows) if rows is None else rows
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_topk_rows(got[rows], p, rows, scores)
    assert not bad, bad[:10]


def causal(p):
    p.starts = np.zeros(p.rows, np.int32)
    p.ends = (p.keys - p.rows + 1 + np.arange(p.rows)).astype(np.int32)
    return p


@pytest.mark.parametrize("seed,rows,keys,topk", [
    (10, 1, 1, 512), (11, 3, 100, 512), (13, 9, 2100, 1024), (14, 40, 5000, 2048), (15, 33, 4097, 512),
    (16, 16, 20000, 1024), (17, 25, 40000, 512), (18, 61, 9000, 1024),
])
def test_fold_random_ranges(mqa, seed, rows, keys, topk):
    """Empty, reversed, short and long ranges; ragged last block of 6 rows."""
    p = synth.random_small(seed, rows, keys, topk)
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0, stats
    assert_parity(p, got)


def test_fold_gated_split_causal(mqa):
    """Long causal rows: sampled gate on fold scores, binned selection, key
    chunks merged across CTAs; every row classified safe."""
    p = causal(synth.random_small(27, 24, 60000, 2048, empty_frac=0.0))
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0, stats
    assert stats["gated_rows"] == 24 and stats["unsafe_rows"] == 0, stats
    assert 0 < stats["fold_bound_ppm"] < 1_000_000, stats
    assert_parity(p, got)


@pytest.mark.parametrize("force_gate", [1, 2])
def test_fold_forced_gate_rescans(mqa, force_gate):
    """Gate at +inf (every row under-fills) or off with a reduced slab (long
    rows overflow): the exact direct rescan gives the top-k."""
    p = synth.random_small(21, 24, 30000, 512, empty_frac=0.0)
    got, status, stats = run(mqa, p, dict(FOLD, force_gate=force_gate, slab_capacity=2560))
    assert status == 0, stats
    assert stats["rows_rescanned"] > 0, stats
    assert_parity(p, got)


def test_fold_forced_unsafe_rescans_every_row(mqa):
    """Every row the fold would serve classified unsafe: all are rescanned
    with the direct head sum, the result is still exact."""
    p = synth.random_small(22, 30, 30000, 1024, empty_frac=0.0)
    got, status, stats = run(mqa, p, dict(FOLD, force_unsafe=1))
    assert status == 0, stats
    n = p.visible()
    assert stats["unsafe_rows"] == int(np.sum(n > p.topk)), stats
    assert stats["rows_rescanned"] >= stats["unsafe_rows"], stats
    assert_parity(p, got)


def relu_dominated(seed, rows, keys, topk, pos_keys, row_len):
    """Rows whose true scores are 0 for almost every key: every query element
    and weight is positive, most keys have every element negative (each head's
    dot product is negative, relu clears it) at scale 1, and pos_keys keys are
    positive at scale 2^-20.  The folded query is large while the top scores
    are tiny, so the fold's error bound exceeds 2^-16 of the row's largest
    |score| by orders of magnitude: the row must be classified unsafe and
    rescanned exactly, or its selection would be decided by rounding."""
    rng = np.random.default_rng(seed)
    q = synth.quantize_e4m3fn(np.abs(rng.standard_normal((rows, synth.HEADS, synth.HEAD_DIM), dtype=np.float32)))
    w = (np.abs(rng.standard_normal((rows, synth.HEADS), dtype=np.float32)) / np.float32(np.sqrt(32))).astype(np.float32)
    kf = -np.abs(rng.standard_normal((keys, synth.HEAD_DIM), dtype=np.float32)) - np.float32(0.25)
    exps = np.full(keys, 127, np.int64)
    pos = rng.choice(keys, size=pos_keys, replace=False)
    kf[pos] = -kf[pos]
    exps[pos] = 107
    k = synth.quantize_e4m3fn(kf)
    starts = rng.integers(0, keys - row_len, size=rows).astype(np.int32)
    ends = (starts + row_len).astype(np.int32)
    return synth.Problem(f"relu_dominated_{seed}", q, k, synth.ue8m0_bytes(exps.astype(np.uint8)), w, starts, ends,
                         topk)


@pytest.mark.parametrize("row_len", [2000, 20000])
def test_fold_relu_dominated_rows_are_unsafe(mqa, row_len):
    """Natural unsafe rows, gated (20000 keys) and ungated (2000 keys, more
    than top-k): classified unsafe, rescanned, exact."""
    p = relu_dominated(31, 18, 40000, 512, 4000, row_len)
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0, stats
    assert stats["unsafe_rows"] == p.rows, stats
    assert stats["fold_bound_ppm"] > 1_000_000, stats
    assert_parity(p, got)


def test_fold_wide_weight_range(mqa):
    """Weights spanning 2^-40 .. 2^40 within a row, and rows scaled by 1e6 and
    1e-6: the bound is relative, so these rows are served by the fold (or
    rescanned); either way the top-k is exact."""
    p = synth.random_small(33, 24, 30000, 1024, empty_frac=0.0)
    rng = np.random.default_rng(1)
    p.weights[0:6] *= np.exp2(rng.integers(-40, 41, size=(6, 32))).astype(np.float32)
    p.weights[6:12] *= np.float32(1e6)
    p.weights[12:18] *= np.float32(1e-6)
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0, stats
    assert_parity(p, got)


def test_fold_full_size_128k(mqa):
    """16,384 rows x 131,072 keys through the fold compilation: every row's
    structure, sampled rows against the oracle, no unsafe row."""
    p = synth.make("r16k_128k_k2048")
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0 and stats["unsafe_rows"] == 0, stats
    rows = synth.sample_rows(p, 40)
    assert_parity(p, got, rows)


def test_fold_adversarial_1m_scaled_rows_are_safe(mqa):
    """The 1M-key adversarial chunk (25% duplicated keys, 1% of weight rows
    scaled by 1e6): the fold's bound is relative to each row's scores, so the
    scaled rows are provably safe (fold_bound_ppm below one million) and every
    one of them is checked against the oracle."""
    p = synth.make("r16k_1m_k2048_adversarial")
    got, status, stats = run(mqa, p, FOLD)
    assert status == 0, stats
    assert stats["unsafe_rows"] == 0 and stats["fold_bound_ppm"] < 1_000_000, stats
    rows = np.unique(np.concatenate([p.special_rows, synth.sample_rows(p, 8)]))
    assert_parity(p, got, rows)
