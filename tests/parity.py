"""Helpers for comparing the CUDA path with the oracle.

Pass rule for top-k (fixed by the target definition: exact top-k up to ties
at the boundary): structure is bit-exact (c = min(topk, n) distinct in-range
relative indices, then -1), a row with n <= topk returns exactly {0..n-1},
and every key in the symmetric difference between the GPU set and the
oracle set has an oracle score within 1e-4 * max|score| of the row's oracle
k-th score.  Logits: |gpu - oracle| <= 1e-3 * max|score| per row, -inf
exactly outside the row's range.
"""
import numpy as np

TOPK_TIE_TOL = 1e-4
LOGITS_TOL = 1e-3


def to_device(p, dev="cuda"):
    import torch
    import sparse_attention_indexer_relu_gb300 as mqa
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q, k = t(p.q), t(p.k)
    scales = mqa.ue8m0_decode(t(p.scales_ue8m0))
    return q, k, scales, t(p.weights), t(p.starts), t(p.ends)


def check_topk_rows(got, p, rows, scores, oracle_idx=None):
    """got: [len(rows), topk] int32 (GPU), scores: oracle fp64 scores [len(rows), keys]."""
    bad = []
    for i, r in enumerate(rows):
        s, e = int(p.starts[r]), int(p.ends[r])
        n = max(0, e - s)
        c = min(p.topk, n)
        g = got[i]
        if not np.all(g[c:] == -1):
            bad.append((r, "padding"))
            continue
        sel = g[:c]
        if np.any(sel < 0) or np.any(sel >= n) or len(np.unique(sel)) != c:
            bad.append((r, "indices"))
            continue
        if n <= p.topk:
            if set(sel.tolist()) != set(range(n)):
                bad.append((r, "short row set"))
            continue
        vis = scores[i, s:e]
        tol = TOPK_TIE_TOL * np.max(np.abs(vis))
        order = np.argsort(-vis, kind="stable")
        kth = vis[order[c - 1]]
        want = set(order[:c].tolist())
        diff = want ^ set(sel.tolist())
        worst = max((abs(vis[j] - kth) for j in diff), default=0.0)
        if worst > tol:
            bad.append((r, f"tie rule: {len(diff)} keys differ, worst |S-kth| = {worst:.3g} > {tol:.3g}"))
    return bad


def check_logits_rows(got, p, rows, scores):
    bad = []
    for i, r in enumerate(rows):
        ref = scores[i]
        fin = np.isfinite(ref)
        if not np.array_equal(np.isneginf(got[i]), ~fin):
            bad.append((r, "-inf pattern"))
            continue
        if fin.any():
            tol = LOGITS_TOL * np.max(np.abs(ref[fin]))
            err = np.max(np.abs(got[i][fin] - ref[fin]))
            if err > tol:
                bad.append((r, f"max err {err:.3g} > {tol:.3g}"))
    return bad


def block_scores(scores_row, s, e):
    """Block scores of a row: the largest oracle score over its visible keys in
    each block of 8 keys, blocks floor(s/8) .. floor((e-1)/8)."""
    if e <= s:
        return np.zeros(0)
    b0 = s // 8
    nb = (e - 1) // 8 - b0 + 1
    out = np.full(nb, -np.inf)
    keys = np.arange(s, e)
    np.maximum.at(out, keys // 8 - b0, scores_row[s:e])
    return out


def check_block_rows(got, p, rows, scores, btopk):
    """got: [len(rows), btopk] block indices relative to floor(start/8) (GPU);
    scores: oracle fp64 key scores.  Same rule as check_topk_rows, on blocks."""
    bad = []
    for i, r in enumerate(rows):
        s, e = int(p.starts[r]), int(p.ends[r])
        bs = block_scores(scores[i], s, e)
        n = len(bs)
        c = min(btopk, n)
        g = got[i]
        if not np.all(g[c:] == -1):
            bad.append((r, "padding"))
            continue
        sel = g[:c]
        if np.any(sel < 0) or np.any(sel >= n) or len(np.unique(sel)) != c:
            bad.append((r, "indices"))
            continue
        if n <= btopk:
            if set(sel.tolist()) != set(range(n)):
                bad.append((r, "short row set"))
            continue
        tol = TOPK_TIE_TOL * np.max(np.abs(bs))
        order = np.argsort(-bs, kind="stable")
        kth = bs[order[c - 1]]
        diff = set(order[:c].tolist()) ^ set(sel.tolist())
        worst = max((abs(bs[j] - kth) for j in diff), default=0.0)
        if worst > tol:
            bad.append((r, f"tie rule: {len(diff)} blocks differ, worst |B-kth| = {worst:.3g} > {tol:.3g}"))
    return bad


def numpy_block_mask(lists, starts, ends, keys, words):
    """Block mask and visible-key counts built on the CPU from block lists
    relative to floor(start / 8) (-1 / out-of-range entries ignored)."""
    rows = lists.shape[0]
    mask = np.zeros((rows, words), np.uint32)
    items = np.zeros(rows, np.int32)
    for r in range(rows):
        s = max(int(starts[r]), 0)
        e = max(s, min(int(ends[r]), keys))
        b0, blast = s // 8, ((e - 1) // 8 if e > s else s // 8 - 1)
        seen = set()
        for rel in lists[r]:
            rel = int(rel)
            if rel < 0 or rel > blast - b0:
                continue
            b = b0 + rel
            if b in seen:
                continue
            seen.add(b)
            mask[r, b // 32] |= np.uint32(1 << (b % 32))
            items[r] += min(e, 8 * b + 8) - max(s, 8 * b)
    return mask, items


def check_masked_rows(got, p, rows, scores):
    """Masked selection: visible keys are those with a finite oracle score."""
    bad = []
    for i, r in enumerate(rows):
        s, e = int(p.starts[r]), int(p.ends[r])
        vis = scores[i, s:e] if e > s else np.zeros(0)
        keep = np.nonzero(np.isfinite(vis))[0]
        c = min(p.topk, len(keep))
        g = got[i]
        if not np.all(g[c:] == -1):
            bad.append((r, "padding"))
            continue
        sel = g[:c]
        if not set(sel.tolist()) <= set(keep.tolist()) or len(np.unique(sel)) != c:
            bad.append((r, "indices"))
            continue
        if len(keep) <= p.topk:
            continue
        v = vis[keep]
        tol = TOPK_TIE_TOL * np.max(np.abs(v))
        order = keep[np.argsort(-v, kind="stable")]
        kth = vis[order[c - 1]]
        diff = set(order[:c].tolist()) ^ set(sel.tolist())
        worst = max((abs(vis[j] - kth) for j in diff), default=0.0)
        if worst > tol:
            bad.append((r, f"tie rule: {len(diff)} keys differ, worst |S-kth| = {worst:.3g} > {tol:.3g}"))
    return bad
