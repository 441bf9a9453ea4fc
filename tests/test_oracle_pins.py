"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check ties the oracle to an independent fact: torch's float8_e4m3fn cast,
exact integer arithmetic, a numpy matmul formulation, closed forms, the
pages' printed rule for UE8M0 scales, a hand-worked example, brute force over
subsets, and invariances of the definition.  `test_oracle_mutations.py` shows
that planted mistakes in the oracle fail these pins.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# independent helpers (torch decode, numpy fp64 formulation)

def torch_decode_e4m3(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def numpy_scores(p, rows=None):
    """Scores from a different formulation: torch decode, fp64 matmul for all
    heads at once, relu(s) = (s + |s|)/2, scale from 2**(e-127) via ldexp."""
    rows = np.arange(p.rows) if rows is None else np.asarray(rows)
    kd = torch_decode_e4m3(p.k)                       # [N, D]
    e = p.scales_ue8m0[:, 0].astype(np.int64)
    scale = np.ldexp(1.0, e - 127)
    out = np.full((len(rows), p.keys), -np.inf)
    for i, r in enumerate(rows):
        qd = torch_decode_e4m3(p.q[r])               # [H, D]
        s = qd @ kd.T                                 # [H, N], exact
        relu = 0.5 * (s + np.abs(s))
        val = scale * (p.weights[r].astype(np.float64) @ relu)
        lo, hi = int(p.starts[r]), int(p.ends[r])
        if hi > lo:
            out[i, lo:hi] = val[lo:hi]
    return out


def tiny_problem(seed, rows, keys, topk, heads=synth.HEADS, dim=synth.HEAD_DIM):
    return synth.random_small(seed, rows, keys, topk, heads=heads, dim=dim)


def check_topk_against_scores(idx_row, scores_row, start, end, topk):
    """idx_row must hold c = min(topk, n) distinct in-range relative indices,
    then -1s, and every selected score must be >= every unselected score."""
    n = max(0, end - start)
    c = min(topk, n)
    assert np.all(idx_row[c:] == -1)
    sel = idx_row[:c]
    assert np.all((sel >= 0) & (sel < n))
    assert len(np.unique(sel)) == c
    if c and c < n:
        vis = scores_row[start:end]
        mask = np.zeros(n, bool)
        mask[sel] = True
        assert vis[mask].min() >= vis[~mask].max()


# ----------------------------------------------------------------------------
# e4m3 table

def test_e4m3_table_matches_torch_cast(lib=None):
    tab = oracle.e4m3_table(lib=lib)
    ref = torch_decode_e4m3(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(tab[~nan], ref[~nan])


def test_e4m3_table_landmarks(lib=None):
    tab = oracle.e4m3_table(lib=lib)
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert tab[0x01] == 2.0 ** -9          # smallest subnormal
    assert tab[0x08] == 2.0 ** -6          # smallest normal
    assert tab[0x38] == 1.0
    pos = tab[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)        # code order is value order
    assert np.all(np.isclose(tab[0x80:0xFF], -tab[0x00:0x7F]) | (tab[0x80:0xFF] == 0))


def test_quantizer_matches_torch_rne(lib=None):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 4,
                        rng.standard_normal(20000).astype(np.float32) * 1e-3,
                        np.float32([0.0, -0.0, 448.0, -448.0, 2 ** -9, 2 ** -10, 3 * 2 ** -10,
                                    1.0625, 1.1875, 300.0, 440.0])])
    mine = synth.quantize_e4m3fn(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(torch_decode_e4m3(mine), torch_decode_e4m3(ref))


def test_quantizer_saturates(lib=None):
    codes = synth.quantize_e4m3fn(np.float32([500.0, -1e4, 449.0]))
    assert codes.tolist() == [0x7E, 0xFE, 0x7E]


# ----------------------------------------------------------------------------
# UE8M0

def test_ue8m0_all_exponents_closed_form(lib=None):
    e = np.arange(256, dtype=np.uint8)
    got = oracle.ue8m0_decode(synth.ue8m0_bytes(e), lib=lib)
    for ei in range(256):
        if ei == 0:
            want = 0.0
        elif ei == 255:
            want = math.inf
        else:
            want = math.ldexp(1.0, ei - 127)
        assert got[ei] == np.float32(want), ei
    # the bit-pattern rule for the whole range
    assert np.array_equal(got.view(np.uint32), e.astype(np.uint32) << 23)


def test_ue8m0_golden_examples(lib=None):
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "ue8m0_examples.txt"))
            if ln.strip() and not ln.startswith("#")]
    e = np.array([int(r[0]) for r in rows], np.uint8)
    got = oracle.ue8m0_decode(synth.ue8m0_bytes(e), lib=lib)
    for (es, val, bits), g in zip(rows, got):
        assert g == np.float32(float(val))
        assert int(np.float32(g).view(np.uint32)) == int(bits, 16)


# ----------------------------------------------------------------------------
# exact dot products (integer brute force)

def test_head_dots_exact_integer_bruteforce(lib=None):
    p = tiny_problem(11, 3, 40, 8)
    # every e4m3 value times 2^9 is an integer
    qi = np.rint(torch_decode_e4m3(p.q) * 512).astype(np.int64)
    ki = np.rint(torch_decode_e4m3(p.k) * 512).astype(np.int64)
    assert np.array_equal(qi / 512.0, torch_decode_e4m3(p.q))
    for r in range(p.rows):
        for j in (0, 7, 39):
            want = [sum(int(a) * int(b) for a, b in zip(qi[r, h], ki[j])) for h in range(p.heads)]
            got = oracle.head_dots(p.q, p.k, r, j, lib=lib)
            assert [int(v) for v in np.rint(np.ldexp(got, 18))] == want
            assert np.array_equal(np.ldexp(np.array(want, dtype=np.float64), -18), got)


def test_head_dots_extreme_codes_exact(lib=None):
    # +-448 everywhere: 128 * 448^2 = 25690112 exactly
    q = np.full((1, 2, 128), 0x7E, np.uint8)
    q[0, 1] = 0xFE
    k = np.full((1, 128), 0x7E, np.uint8)
    got = oracle.head_dots(q, k, 0, 0, lib=lib)
    assert got.tolist() == [128 * 448.0 ** 2, -128 * 448.0 ** 2]


# ----------------------------------------------------------------------------
# scores: independent formulation

@pytest.mark.parametrize("seed", [1, 2])
def test_scores_match_numpy_formulation(seed, lib=None):
    p = tiny_problem(seed, 12, 700, 64)
    _, s = oracle.run(p, want_topk=False, want_scores=True, lib=lib)
    ref = numpy_scores(p)
    assert np.array_equal(np.isinf(s), np.isinf(ref))
    fin = np.isfinite(ref)
    rowmax = np.max(np.where(fin, np.abs(ref), 0), axis=1, keepdims=True) + 1e-300
    diff = np.abs(np.where(fin, s, 0.0) - np.where(fin, ref, 0.0))
    assert np.all(diff <= 1e-12 * rowmax)


def test_hand_example_golden(lib=None):
    vals = {}
    for ln in open(os.path.join(GOLDEN, "hand_example.txt")):
        if ln.strip() and not ln.startswith("#"):
            parts = ln.split()
            vals[parts[0]] = parts[1:]
    q = np.array([int(x, 16) for x in vals["q"]], np.uint8).reshape(1, 2, 2)
    k = np.array([int(x, 16) for x in vals["k"]], np.uint8).reshape(5, 2)
    w = np.array([float(x) for x in vals["w"]], np.float32).reshape(1, 2)
    e = np.array([int(x) for x in vals["e"]], np.uint8)
    s0, e0 = (int(x) for x in vals["range"])
    tk = int(vals["topk"][0])
    p = synth.Problem("hand", q, k, synth.ue8m0_bytes(e), w, np.int32([s0]), np.int32([e0]), tk)
    idx, sc = oracle.run(p, want_scores=True, lib=lib)
    assert sc[0, s0:e0].tolist() == [float(x) for x in vals["scores"]]
    assert np.isneginf(sc[0, 0])
    assert idx[0].tolist() == [int(x) for x in vals["expected"]]


# ----------------------------------------------------------------------------
# special case that reduces to a library routine: one head, positive weight

def test_single_head_reduces_to_gemv_topk(lib=None):
    p = tiny_problem(21, 6, 3000, 100)
    p.weights[:] = 0
    p.weights[:, 5] = 1.0
    p.starts[:] = 0
    p.ends[:] = p.keys
    p.scales_ue8m0[:] = 127  # unit scales
    idx = oracle.topk(p, lib=lib)
    kd = torch_decode_e4m3(p.k)
    for r in range(p.rows):
        g = torch_decode_e4m3(p.q[r, 5]) @ kd.T
        g = np.maximum(g, 0)
        part = np.argpartition(-g, p.topk - 1)[: p.topk]
        kth = np.sort(g)[::-1][p.topk - 1]
        # same multiset of selected values; sets agree off the kth value
        assert np.array_equal(np.sort(g[idx[r]]), np.sort(g[part]))
        assert set(idx[r][g[idx[r]] > kth]) == set(part[g[part] > kth])


# ----------------------------------------------------------------------------
# brute force over subsets on tiny rows

def test_bruteforce_subsets_tiny_rows(lib=None):
    rng = np.random.default_rng(3)
    for trial in range(30):
        n = int(rng.integers(1, 10))
        keys = n + 3
        topk = int(rng.integers(1, n + 3))
        p = tiny_problem(100 + trial, 1, keys, topk, heads=4, dim=8)
        p.starts[:] = 2
        p.ends[:] = 2 + n if 2 + n <= keys else keys
        n = int(p.ends[0] - p.starts[0])
        idx, _ = oracle.run(p, lib=lib)
        sc = numpy_scores(p)[0, 2:2 + n]
        c = min(topk, n)
        best = max(itertools.combinations(range(n), c), key=lambda s: (sum(sc[list(s)]), [-x for x in s]))
        got = sorted(idx[0, :c].tolist())
        assert np.isclose(sum(sc[got]), sum(sc[list(best)]), rtol=0, atol=1e-12 * (1 + np.abs(sc).sum()))
        check_topk_against_scores(idx[0], np.concatenate([np.zeros(2), sc]), 2, 2 + n, topk)


# ----------------------------------------------------------------------------
# structure: padding, relative indices, short rows

@pytest.mark.parametrize("n", [0, 1, 511, 512, 513, 700])
def test_row_lengths_around_topk(n, lib=None):
    p = tiny_problem(7, 2, 800, 512)
    p.starts[:] = [50, 0]
    p.ends[:] = [50 + n, n]
    idx, sc = oracle.run(p, want_scores=True, lib=lib)
    for r in range(2):
        check_topk_against_scores(idx[r], sc[r], int(p.starts[r]), int(p.ends[r]), 512)
        if n <= 512:
            assert sorted(idx[r, :n].tolist()) == list(range(n))


def test_reversed_range_is_empty(lib=None):
    p = tiny_problem(8, 1, 100, 16)
    p.starts[:] = 60
    p.ends[:] = 20
    idx = oracle.topk(p, lib=lib)
    assert np.all(idx == -1)


def test_out_of_range_rejected(lib=None):
    p = tiny_problem(9, 1, 100, 16)
    p.starts[:] = 10
    p.ends[:] = 101
    with pytest.raises(ValueError):
        oracle.topk(p, lib=lib)


# ----------------------------------------------------------------------------
# invariances of the definition

def test_invariant_key_permutation_in_window(lib=None):
    p = tiny_problem(31, 4, 900, 64)
    p.starts[:] = 100
    p.ends[:] = 800
    base = oracle.topk(p, lib=lib)
    rng = np.random.default_rng(0)
    perm = rng.permutation(700)
    p2 = synth.Problem("perm", p.q, p.k.copy(), p.scales_ue8m0.copy(), p.weights, p.starts, p.ends, p.topk)
    p2.k[100:800] = p.k[100:800][perm]
    p2.scales_ue8m0[100:800] = p.scales_ue8m0[100:800][perm]
    got = oracle.topk(p2, lib=lib)
    inv = np.argsort(perm)  # new position of old key t is inv[t]
    for r in range(p.rows):
        assert set(got[r].tolist()) == set(inv[base[r]].tolist())


def test_invariant_power_of_two_scale(lib=None):
    p = tiny_problem(32, 3, 600, 50)
    _, s = oracle.run(p, want_scores=True, lib=lib)
    p2 = synth.Problem("x2", p.q, p.k, p.scales_ue8m0 + 3, p.weights, p.starts, p.ends, p.topk)
    idx2, s2 = oracle.run(p2, want_scores=True, lib=lib)
    assert np.array_equal(s2, s * 8.0)
    assert np.array_equal(idx2, oracle.topk(p, lib=lib))


def test_invariant_shift_with_prepended_keys(lib=None):
    p = tiny_problem(33, 3, 500, 40)
    base = oracle.topk(p, lib=lib)
    pad = 77
    k2 = np.concatenate([np.full((pad, p.dim), 0x38, np.uint8), p.k])
    g2 = np.concatenate([np.full((pad, 4), 127, np.uint8), p.scales_ue8m0])
    p2 = synth.Problem("shift", p.q, k2, g2, p.weights, p.starts + pad, p.ends + pad, p.topk)
    assert np.array_equal(oracle.topk(p2, lib=lib), base)


def test_tiny_config_structure(lib=None):
    p = synth.make("tiny_64x4096_k512")
    idx, sc = oracle.run(p, want_scores=True, lib=lib)
    for r in range(p.rows):
        check_topk_against_scores(idx[r], sc[r], int(p.starts[r]), int(p.ends[r]), p.topk)


def test_dense_budget_table_golden(lib=None):
    """The dense baseline's chunking rule (rows per call = 2**27 / keys under a
    512 MiB fp32 budget) and byte model reproduce the pages' table."""
    from sparse_attention_indexer_relu_gb300 import plan
    for ln in open(os.path.join(GOLDEN, "dense_logits_budget.txt")):
        if not ln.strip() or ln.startswith("#"):
            continue
        keys, gib, calls, traffic = ln.split()
        keys = int(keys)
        assert plan.dense_logits_bytes(16384, keys) == int(gib) * 2 ** 30
        assert plan.dense_logits_traffic_bytes(16384, keys) == int(traffic) * 2 ** 30
        if calls != "-":
            assert plan.dense_calls(16384, keys, 512 * 2 ** 20) == int(calls)


def test_fast_quantizer_matches_reference(lib=None):
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(300000).astype(np.float32) * 3,
                        np.float32([1000.0, -700.0, 449.0, 2 ** -12, -2 ** -9])])
    assert np.array_equal(synth.quantize_e4m3fn_fast(x), synth.quantize_e4m3fn(x))


# ----------------------------------------------------------------------------
# block selection (two-level candidate selection): blocks of 8 keys ranked by
# their largest score

def check_blocks_against_scores(blk_row, scores_row, start, end, btopk, tol):
    """blk_row must hold c = min(btopk, nb) distinct block indices relative to
    floor(start / 8), then -1s, and every selected block's largest score must
    be >= every unselected block's (up to tol)."""
    b0 = start // 8
    nb = ((end - 1) // 8 - b0 + 1) if end > start else 0
    c = min(btopk, nb)
    assert np.all(blk_row[c:] == -1)
    sel = blk_row[:c]
    assert np.all((sel >= 0) & (sel < nb)) and len(np.unique(sel)) == c
    if c and c < nb:
        bmax = np.full(nb, -np.inf)
        for j in range(start, end):
            b = j // 8 - b0
            bmax[b] = max(bmax[b], scores_row[j])
        mask = np.zeros(nb, bool)
        mask[sel] = True
        assert bmax[mask].min() >= bmax[~mask].max() - tol


@pytest.mark.parametrize("seed", [7, 8])
def test_blocks_match_numpy_formulation(seed, lib=None):
    """Block maxima from the independent numpy scores rank the oracle's blocks."""
    p = tiny_problem(seed, 12, 900, 64)
    blk = oracle.run_blocks(p, 40, lib=lib)
    sc = numpy_scores(p)
    for r in range(p.rows):
        tol = 1e-9 * (1 + np.abs(sc[r][np.isfinite(sc[r])]).max(initial=0))
        check_blocks_against_scores(blk[r], sc[r], int(p.starts[r]), int(p.ends[r]), 40, tol)


def test_blocks_reduce_to_key_topk_on_sparse_blocks(lib=None):
    """Keys 8b+1 .. 8b+7 are zero vectors (score 0) and every other score is
    positive, so block b's score is key 8b's: the block selection must equal
    the key selection over the keys 8b alone (same scores, same tie rule)."""
    p = tiny_problem(9, 6, 1600, 64, heads=8, dim=32)
    p.q = (p.q & 0x7F).astype(np.uint8)              # non-negative q
    p.k = (p.k & 0x7F).astype(np.uint8)              # non-negative k
    p.weights = np.abs(p.weights).astype(np.float32) + np.float32(1e-3)
    zero = np.arange(p.keys) % 8 != 0
    p.k[zero] = 0
    p.starts = (p.starts // 8 * 8).astype(np.int32)
    p.ends = (p.ends // 8 * 8).astype(np.int32)
    blk = oracle.run_blocks(p, 32, lib=lib)
    sub = synth.Problem("sub", p.q, p.k[::8].copy(), p.scales_ue8m0[::8].copy(), p.weights,
                        (p.starts // 8).astype(np.int32), (p.ends // 8).astype(np.int32), 32)
    idx, _ = oracle.run(sub, lib=lib)
    assert np.array_equal(blk, idx)


def test_blocks_integer_bruteforce_tiny(lib=None):
    """Exact block maxima from Python integers (codes decoded by hand, dots in
    units of 2^-18, one head, unit weight, scale 1) on tiny rows."""
    def dec(c):
        s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
        v = (m if e == 0 else (8 + m) << (e - 1))     # value * 2^9
        return -v if s else v
    rng = np.random.default_rng(4)
    for trial in range(20):
        keys = int(rng.integers(9, 60))
        p = tiny_problem(200 + trial, 1, keys, 8, heads=1, dim=4)
        p.weights[:] = 1.0
        p.scales_ue8m0[:] = 127
        s0 = int(rng.integers(0, keys - 1))
        p.starts[:] = s0
        p.ends[:] = int(rng.integers(s0 + 1, keys + 1))
        st, en = int(p.starts[0]), int(p.ends[0])
        qd = [dec(int(c)) for c in p.q[0, 0]]
        score = {j: max(0, sum(a * dec(int(b)) for a, b in zip(qd, p.k[j]))) for j in range(st, en)}
        b0 = st // 8
        bmax = {}
        for j, v in score.items():
            bmax[j // 8 - b0] = max(bmax.get(j // 8 - b0, -1), v)
        want = sorted(bmax, key=lambda b: (-bmax[b], b))[:5]
        got = oracle.run_blocks(p, 5, lib=lib)[0]
        assert got[:len(want)].tolist() == want
        assert np.all(got[len(want):] == -1)


# ----------------------------------------------------------------------------
# masked selection (the consumer half of the two-level selection)

def random_block_mask(rng, rows, keys, frac):
    words = (keys + 255) // 256
    bits = rng.random((rows, words * 32)) < frac
    return np.packbits(bits.reshape(rows, words, 32)[:, :, ::-1], axis=-1).view(">u4").reshape(rows, words) \
        .astype(np.uint32)


def allowed_keys(mask_row, keys):
    j = np.arange(keys)
    return ((mask_row[j >> 8] >> ((j >> 3) & 31)) & 1).astype(bool)


def test_masked_full_mask_is_unmasked(lib=None):
    p = tiny_problem(60, 9, 2000, 64)
    full = np.full((p.rows, (p.keys + 255) // 256), 0xFFFFFFFF, np.uint32)
    a, _ = oracle.run_masked(p, full, lib=lib)
    b, _ = oracle.run(p, lib=lib)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("frac", [0.1, 0.6])
def test_masked_matches_numpy_formulation(frac, lib=None):
    """Allowed keys from an independent bit decode, scores from the numpy
    formulation: the masked selection is the top-k over the allowed keys."""
    rng = np.random.default_rng(61)
    p = tiny_problem(61, 10, 2500, 48)
    mask = random_block_mask(rng, p.rows, p.keys, frac)
    idx, _ = oracle.run_masked(p, mask, lib=lib)
    sc = numpy_scores(p)
    for r in range(p.rows):
        s, e = int(p.starts[r]), int(p.ends[r])
        allow = allowed_keys(mask[r], p.keys)
        vis = np.full(p.keys, -np.inf)
        vis[allow] = sc[r][allow]
        keep = np.nonzero(allow[s:e])[0]            # visible relative indices
        c = min(48, len(keep))
        sel = idx[r][:c]
        assert np.all(idx[r][c:] == -1)
        assert set(sel.tolist()) <= set(keep.tolist()) and len(np.unique(sel)) == c
        if 0 < c < len(keep):
            rest = np.setdiff1d(keep, sel)
            assert vis[s + sel].min() >= vis[s + rest].max() - 1e-9 * (1 + np.abs(sc[r][np.isfinite(sc[r])]).max())


def test_masked_integer_bruteforce_tiny(lib=None):
    def dec(c):
        s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
        v = (m if e == 0 else (8 + m) << (e - 1))
        return -v if s else v
    rng = np.random.default_rng(62)
    for trial in range(20):
        keys = int(rng.integers(20, 120))
        p = tiny_problem(300 + trial, 1, keys, 6, heads=1, dim=4)
        p.weights[:] = 1.0
        p.scales_ue8m0[:] = 127
        p.starts[:] = 0
        p.ends[:] = keys
        mask = random_block_mask(rng, 1, keys, 0.5)
        allow = allowed_keys(mask[0], keys)
        qd = [dec(int(c)) for c in p.q[0, 0]]
        score = {j: max(0, sum(a * dec(int(b)) for a, b in zip(qd, p.k[j]))) for j in range(keys) if allow[j]}
        want = sorted(score, key=lambda j: (-score[j], j))[:6]
        got, _ = oracle.run_masked(p, mask, topk=6, lib=lib)
        assert got[0][:len(want)].tolist() == want
        assert np.all(got[0][len(want):] == -1)


# ---------------------------------------------------------------- the fold (relu(s) = (s + |s|) / 2)
def _e4m3_values(lib=None):
    return oracle.e4m3_table(lib=lib)


def test_e4m3_encode_is_torch_round_to_nearest_even(lib=None):
    """The oracle's encoder (search over the table) against torch's float8_e4m3fn
    cast, an independent RNE implementation, on random values, every halfway
    point between adjacent codes, subnormals and signed zeros."""
    tab = _e4m3_values(lib)
    pos = np.sort(tab[:0x7F])
    halves = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(90)
    xs = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-2, 2, 2000), rng.uniform(-0.02, 0.02, 1000),
                         halves, -halves, pos, -pos, [0.0, -0.0, 448.0, -448.0]]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x), lib=lib) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_fold_query_is_the_weighted_head_sum(lib=None):
    """v = sum_h w_h E(q_h) formed in fp32: within fp32 rounding of the exact fp64 sum."""
    p = synth.random_small(91, 12, 100, 512)
    _, _, v, _ = oracle.fold_prep(p.q, p.weights, lib=lib)
    tab = _e4m3_values(lib)
    qd = tab[p.q.astype(np.int64)]                       # [rows, heads, dim]
    exact = np.einsum("rh,rhd->rd", p.weights.astype(np.float64), qd)
    bound = 32 * 2.0 ** -24 * np.einsum("rh,rhd->rd", np.abs(p.weights.astype(np.float64)), np.abs(qd))
    assert np.all(np.abs(v.astype(np.float64) - exact) <= bound + 1e-30)


def test_fold_terms_reconstruct_and_are_minimal(lib=None):
    """sum_t 2^e_t E(u_t) plus the residual rebuilds v exactly; every term's
    exponent is the smallest that keeps its scaled residual within 448; beta is
    the residual's 2-norm; with 4 terms the residual is below 2^-16 of v."""
    tab = _e4m3_values(lib)
    for seed in (92, 93):
        p = synth.random_small(seed, 16, 100, 512)
        p.weights[3] *= 1e6
        p.weights[5] *= 1e-6
        codes, exps, v, beta = oracle.fold_prep(p.q, p.weights, lib=lib)
        for r in range(p.rows):
            res = v[r].astype(np.float64)
            for t in range(codes.shape[1]):
                m = np.abs(res).max()
                e = int(exps[r, t])
                if m > 0:
                    assert m * 2.0 ** -e <= 448 < m * 2.0 ** -(e - 1)
                term = tab[codes[r, t].astype(np.int64)]
                assert np.all(np.isfinite(term)) and np.abs(term).max() <= 448
                res = res - np.ldexp(term, e)
            assert math.isclose(np.linalg.norm(res), beta[r], rel_tol=1e-12, abs_tol=1e-300)
            assert beta[r] <= 2.0 ** -16 * np.linalg.norm(v[r].astype(np.float64)) + 1e-300


def test_fold_score_identity_and_error_bound(lib=None):
    """The fold's score equals the definition's up to the residual: the
    identity scale * (v_exact . k + sum_h w_h |s_h|) / 2 = S holds in fp64, and
    |S_fold - S| <= scale * beta * |k|_2 / 2 plus the fp32 rounding of v."""
    p = synth.random_small(94, 6, 400, 512, empty_frac=0.0)
    p.starts[:] = 0
    p.ends[:] = p.keys
    codes, exps, v, beta = oracle.fold_prep(p.q, p.weights, lib=lib)
    _, scores = oracle.run(p, want_topk=False, want_scores=True, lib=lib)
    tab = _e4m3_values(lib)
    qd = tab[p.q.astype(np.int64)]
    kd = tab[p.k.astype(np.int64)]
    scale = oracle.ue8m0_decode(p.scales_ue8m0, lib=lib).astype(np.float64)
    w64 = p.weights.astype(np.float64)
    v_exact = np.einsum("rh,rhd->rd", w64, qd)
    s_heads = np.einsum("rhd,jd->rjh", qd, kd)
    ident = scale[None, :] * 0.5 * (v_exact @ kd.T + np.einsum("rh,rjh->rj", w64, np.abs(s_heads)))
    assert np.allclose(ident, scores, rtol=1e-12, atol=1e-12 * np.abs(scores).max())
    rng = np.random.default_rng(95)
    knorm = np.linalg.norm(kd, axis=1)
    vround = np.linalg.norm(v.astype(np.float64) - v_exact, axis=1)
    for _ in range(60):
        r, j = int(rng.integers(p.rows)), int(rng.integers(p.keys))
        f = oracle.fold_score(p, codes, exps, r, j, lib=lib)
        bound = scale[j] * 0.5 * (beta[r] + vround[r]) * knorm[j] * (1 + 1e-9) + 1e-12 * abs(scores[r, j])
        assert abs(f - scores[r, j]) <= bound, (r, j)
