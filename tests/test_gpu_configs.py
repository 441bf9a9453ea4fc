"""Parity on the workload table's chunk shapes, in the launch configuration
the benchmark times: every row is checked for structure, sampled rows against
the oracle (exact top-k up to boundary ties)."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_block_rows, check_masked_rows, check_topk_rows, numpy_block_mask, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mqa():
    import torch
    assert torch.cuda.is_available()
    import sparse_attention_indexer_relu_gb300 as m
    m.lib()
    return m


def structure_all_rows(got, p):
    n = np.maximum(p.ends.astype(np.int64) - p.starts.astype(np.int64), 0)
    c = np.minimum(n, p.topk)
    col = np.arange(p.topk)[None, :]
    valid = col < c[:, None]
    assert np.all(got[~valid] == -1), "padding"
    g = np.where(valid, got, -1)
    assert np.all((g[valid] >= 0) & (g[valid] < np.broadcast_to(n[:, None], g.shape)[valid])), "range"
    srt = np.sort(np.where(valid, got, -1 - col), axis=1)
    assert np.all(np.diff(srt, axis=1) != 0), "duplicates"


CASES = [
    ("r2048_32k_k512", 64),
    ("r2048_32k_k2048", 64),
    ("r16k_128k_k2048", 64),
    ("r16k_128k_k2048_offset4", 64),
    ("multi4_r16k_k1024", 64),
    ("r16k_1m_k2048", 64),
    ("r16k_1m_k2048_adversarial", 64),
    ("decode_b32_s8_64k_k2048", 64),
    ("decode_b4_s8_256k_k2048", 32),
    ("decode_b64_s8_mixed_k512", 64),
    ("h64_r2048_64k_k2048", 64),
]


def checked_rows(p, nsample):
    """Rows checked against the oracle: the sample (evenly spaced rows, every
    row seeing fewer than top-k keys), every specially treated row (the
    adversarial variant's 1e6-scaled weight rows), and every row of the first
    two and the last two 8-row blocks: in causal chunks the lightest blocks
    (rows 0-15) are the ones the key-range split cuts into chunks, the heaviest
    (the last 16 rows) are scanned whole."""
    rows = [synth.sample_rows(p, nsample), p.special_rows]
    if p.rows >= 64:
        rows += [np.arange(16), np.arange(p.rows - 16, p.rows)]
    return np.unique(np.concatenate(rows).astype(np.int64))


@pytest.mark.parametrize("name,nsample", CASES)
def test_config_parity(mqa, name, nsample):
    p = synth.make(name)
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows, heads=p.heads)
    out = mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk, workspace=ws)
    status, stats = mqa.get_status(ws)
    got = out.cpu().numpy()
    assert status == 0, stats
    structure_all_rows(got, p)
    rows = checked_rows(p, nsample)
    if name.startswith("multi4"):
        # every padded row of the 300-key request plus the samples
        rows = np.unique(np.concatenate([rows, np.arange(64)]))
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_topk_rows(got[rows], p, rows, scores)
    assert not bad, (bad[:5], stats)
    print(name, stats)


@pytest.mark.parametrize("name", ["r2048_32k_k2048", "r16k_128k_k2048"])
def test_config_dense_agrees(mqa, name):
    p = synth.make(name)
    q, k, sc, w, s, e = to_device(p)
    dense = mqa.mqa_topk_dense_baseline(q, k, sc, w, s, e, p.topk).cpu().numpy()
    structure_all_rows(dense, p)
    rows = synth.sample_rows(p, 24)
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_topk_rows(dense[rows], p, rows, scores)
    assert not bad, bad[:5]


def structure_blocks(got, p, btopk):
    """Every row's block list: min(btopk, row's blocks) distinct in-range
    indices (relative to floor(start / 8)), then -1."""
    s = p.starts.astype(np.int64)
    e = p.ends.astype(np.int64)
    nb = np.where(e > s, (e - 1) // 8 - s // 8 + 1, 0)
    c = np.minimum(nb, btopk)
    col = np.arange(btopk)[None, :]
    valid = col < c[:, None]
    assert np.all(got[~valid] == -1), "padding"
    assert np.all((got[valid] >= 0) & (got[valid] < np.broadcast_to(nb[:, None], got.shape)[valid])), "range"
    srt = np.sort(np.where(valid, got, -1 - col), axis=1)
    assert np.all(np.diff(srt, axis=1) != 0), "duplicates"


@pytest.mark.parametrize("name,nsample", [("r16k_128k_k2048", 24), ("r16k_1m_k2048", 10)])
def test_config_two_level_parity(mqa, name, nsample):
    """Both stages of the two-level selection on the workload's full chunk:
    the top 2048 blocks of 8 keys (every row's structure, sampled rows against
    the oracle), then the top 512 keys inside seeded random block lists of
    2048 blocks per row (mask built by the GPU kernel for the launch and on
    the CPU for the oracle; sampled rows against the oracle)."""
    import torch
    p = synth.make(name)
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows)
    blk = mqa.mqa_block_topk_prefill(q, k, sc, w, s, e, 2048, workspace=ws)
    status, stats = mqa.get_status(ws)
    assert status == 0, stats
    got_b = blk.cpu().numpy()
    structure_blocks(got_b, p, 2048)
    rows = synth.sample_rows(p, nsample)
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_block_rows(got_b[rows], p, rows, scores, 2048)
    assert not bad, (bad[:5], stats)
    del scores
    # consumer stage on seeded block lists
    rng = np.random.default_rng(80)
    nb = np.maximum((p.ends.astype(np.int64) - 1) // 8 - p.starts.astype(np.int64) // 8 + 1, 1)
    lists = (rng.random((p.rows, 2048)) * nb[:, None]).astype(np.int32)
    words = ((p.keys + 1023) // 1024) * 4
    mask, items = mqa.block_mask(torch.from_numpy(lists).cuda(), s, e, p.keys, words)
    out = mqa.mqa_topk_prefill_masked(q, k, sc, w, s, e, mask, items, 512, workspace=ws)
    status, stats = mqa.get_status(ws)
    assert status == 0, stats
    got_m = out.cpu().numpy()
    cpu_mask, cpu_items = numpy_block_mask(lists[rows], p.starts[rows], p.ends[rows], p.keys, words)
    assert np.array_equal(items.cpu().numpy()[rows], cpu_items)
    sub = synth.Problem(p.name, p.q[rows], p.k, p.scales_ue8m0, p.weights[rows], p.starts[rows], p.ends[rows], 512)
    _, scores = oracle.run_masked(sub, cpu_mask, want_topk=False, want_scores=True)
    bad = check_masked_rows(got_m[rows], sub, np.arange(len(rows)), scores)
    assert not bad, (bad[:5], stats)
    print(name, stats)
