"""Parity of the CUDA path (through the C ABI) with the CPU oracle."""
import numpy as np
import pytest

import oracle
import synth
from parity import (check_block_rows, check_logits_rows, check_masked_rows, check_topk_rows, numpy_block_mask,
                    to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mqa():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_attention_indexer_relu_gb300 as m
    m.lib()
    return m


def run_fused(mqa, p, debug=None, workspace=None):
    import torch
    q, k, sc, w, s, e = to_device(p)
    ws = workspace if workspace is not None else mqa.alloc_workspace(p.rows, heads=p.heads)
    out = mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk, workspace=ws, debug=debug)
    status, stats = mqa.get_status(ws)
    return out.cpu().numpy(), status, stats


def assert_parity(p, got, rows=None):
    rows = np.arange(p.rows) if rows is None else rows
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_topk_rows(got[rows], p, rows, scores)
    assert not bad, bad[:10]


# ---------------------------------------------------------------- workspace
def test_workspace_bytes_for_a_16k_row_chunk(mqa):
    """The fixed workspace of a 16,384-row chunk: per-SM slab slots plus the
    key-range split's slab.  On a 152-SM GB300 it stays within 330 MB."""
    import ctypes
    import torch
    n = ctypes.c_size_t(0)
    assert mqa.lib().mqa_topk_workspace_bytes(0, 16384, ctypes.byref(n)) == 0
    assert n.value > 0
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert n.value <= 330 * 10 ** 6, n.value


# ---------------------------------------------------------------- UE8M0 decode
@pytest.mark.parametrize("keys", [1, 3, 256, 1001, 65536 + 5])
def test_ue8m0_decode_bit_exact(mqa, keys):
    import torch
    rng = np.random.default_rng(keys)
    e = rng.integers(0, 256, size=keys).astype(np.uint8)
    e[: min(keys, 256)] = np.arange(min(keys, 256), dtype=np.uint8)
    g = synth.ue8m0_bytes(e)
    got = mqa.ue8m0_decode(torch.from_numpy(g).cuda()).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), oracle.ue8m0_decode(g).view(np.uint32))


# ---------------------------------------------------------------- debug logits
@pytest.mark.parametrize("name", ["tiny_64x4096_k512"])
def test_logits_debug_config(mqa, name):
    p = synth.make(name)
    q, k, sc, w, s, e = to_device(p)
    got = mqa.mqa_logits_debug(q, k, sc, w, s, e).cpu().numpy()
    _, scores = oracle.run(p, want_topk=False, want_scores=True)
    bad = check_logits_rows(got, p, np.arange(p.rows), scores)
    assert not bad, bad[:10]


@pytest.mark.parametrize("seed,rows,keys", [(1, 1, 1), (2, 5, 130), (3, 17, 999), (4, 40, 5000), (5, 9, 128)])
def test_logits_debug_random(mqa, seed, rows, keys):
    p = synth.random_small(seed, rows, keys, 512)
    q, k, sc, w, s, e = to_device(p)
    got = mqa.mqa_logits_debug(q, k, sc, w, s, e).cpu().numpy()
    _, scores = oracle.run(p, want_topk=False, want_scores=True)
    bad = check_logits_rows(got, p, np.arange(p.rows), scores)
    assert not bad, bad[:10]


# ---------------------------------------------------------------- fused top-k
def test_fused_tiny_config(mqa):
    p = synth.make("tiny_64x4096_k512")
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert_parity(p, got)


@pytest.mark.parametrize("seed,rows,keys,topk", [
    (10, 1, 1, 512), (11, 3, 100, 512), (12, 8, 600, 512), (13, 9, 2100, 1024), (14, 40, 5000, 2048),
    (15, 33, 4097, 512), (16, 16, 20000, 1024), (17, 25, 40000, 512),
])
def test_fused_random_ranges(mqa, seed, rows, keys, topk):
    p = synth.random_small(seed, rows, keys, topk)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert_parity(p, got)


@pytest.mark.parametrize("force_gate", [1, 2])
def test_fused_forced_gate_rescans(mqa, force_gate):
    """Gate forced to +inf (every row under-fills) or off (long rows overflow
    a reduced slab): the exact rescan must still give the exact top-k."""
    p = synth.random_small(21, 24, 30000, 512, empty_frac=0.0)
    got, status, stats = run_fused(mqa, p, debug={"force_gate": force_gate, "slab_capacity": 2560})
    assert status == 0, stats
    assert stats["rows_rescanned"] > 0
    if force_gate == 2:
        assert stats["compactions"] > 0
    assert_parity(p, got)


def test_fused_small_slab_compaction_ties(mqa):
    """Many exact ties (duplicated keys) with a small slab: compaction keeps
    exactly top-k and the tie rule holds."""
    p = synth.random_small(22, 16, 20000, 1024, empty_frac=0.0)
    rng = np.random.default_rng(0)
    dst = rng.choice(p.keys, p.keys // 2, replace=False)
    src = rng.integers(0, 64, size=dst.size)
    p.k[dst] = p.k[src]
    p.scales_ue8m0[dst] = p.scales_ue8m0[src]
    got, status, stats = run_fused(mqa, p, debug={"force_gate": 2, "slab_capacity": 4608})
    assert status == 0, stats
    assert_parity(p, got)


def test_fused_gated_logbin_selection(mqa):
    """Rows longer than a reduced slab are gated; their top-k comes from the
    two-pass log-bin selection (threshold bin gathered in shared memory)."""
    p = synth.random_small(25, 48, 30000, 512, empty_frac=0.0)
    got, status, stats = run_fused(mqa, p, debug={"slab_capacity": 4096})
    assert status == 0, stats
    assert stats["gated_rows"] > 0
    assert stats["select_fallback"] == 0, stats
    assert_parity(p, got)


def test_fused_gated_tie_groups_take_fallback(mqa):
    """Every key is a copy of one of 16 source keys (2048 copies each), so a
    gated row's k-th score sits inside a tie group larger than the selection
    warp's shared-memory list: the slab-pass radix select must take over and
    still return an exact top-k under the tie rule."""
    rows, keys, topk = 16, 32768, 2048
    p = synth.random_small(26, rows, keys, topk, empty_frac=0.0)
    src = np.repeat(np.arange(16), keys // 16)
    np.random.default_rng(5).shuffle(src)
    p.k = p.k[src].copy()
    p.scales_ue8m0 = p.scales_ue8m0[src].copy()
    p.starts = np.zeros(rows, np.int32)
    p.ends = (keys - np.arange(rows)).astype(np.int32)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert stats["gated_rows"] == rows
    assert stats["select_fallback"] > 0, stats
    assert_parity(p, got)


def _causal(p, keys):
    p.starts = np.zeros(p.rows, np.int32)
    p.ends = (keys - p.rows + 1 + np.arange(p.rows)).astype(np.int32)
    return p


def test_fused_key_split_few_blocks(mqa):
    """Three row blocks on a GPU with many more SMs: each block's key range is
    cut into chunks scanned by different CTAs, which share one sampled gate;
    the CTA that finishes a block's last chunk selects over every chunk's
    candidates.  The result must be the exact top-k."""
    p = _causal(synth.random_small(27, 24, 60000, 2048, empty_frac=0.0), 60000)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert stats["split_blocks"] == 3, stats
    assert stats["gated_rows"] == 24 and stats["rows_rescanned"] == 0, stats
    # few blocks per CTA: the compilation whose parked epilogue warps select
    # rows in pairs took part in the selection
    assert stats["pair_rows"] > 0, stats
    assert_parity(p, got)


def test_fused_key_split_ungated_rows(mqa):
    """Split blocks whose rows see too few keys to be gated (at most twice the
    gate's target, 6144 at top-2048): every chunk emits all its keys, the merge
    selects exactly."""
    p = _causal(synth.random_small(28, 16, 12000, 2048, empty_frac=0.0), 12000)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert stats["split_blocks"] == 2 and stats["gated_rows"] == 0, stats
    assert_parity(p, got)


def test_fused_key_split_overflow_rescans(mqa):
    """No gate and a reduced slab on 4 CTAs (2 blocks of 2 key chunks each):
    every chunk's segments overflow, the merging CTA queues the block for an
    exact whole-block rescan."""
    p = _causal(synth.random_small(29, 16, 40000, 512, empty_frac=0.0), 40000)
    got, status, stats = run_fused(mqa, p, debug={"force_gate": 2, "slab_capacity": 2560, "max_ctas": 4})
    assert status == 0, stats
    assert stats["split_blocks"] == 2 and stats["rows_rescanned"] > 0, stats
    assert_parity(p, got)


@pytest.mark.parametrize("force_gate", [0, 1])
def test_fused_spread_merge_two_groups(mqa, force_gate):
    """Four row blocks on 16 CTAs: every block is cut into 4 key chunks, fewer
    than its 8 rows, so each chunk's CTA merges its rows with two groups of 8
    epilogue warps side by side.  With the gate forced to +inf every row
    under-fills, and the rows the groups fail go to the exact rescan.  Either
    way the result must be the exact top-k."""
    p = _causal(synth.random_small(30, 32, 40000, 512, empty_frac=0.0), 40000)
    got, status, stats = run_fused(mqa, p, debug={"force_gate": force_gate, "max_ctas": 16})
    assert status == 0, stats
    assert stats["split_blocks"] == 4, stats
    assert stats["pair_rows"] >= 32, stats
    if force_gate:
        assert stats["rows_rescanned"] == 32, stats
    else:
        assert stats["gated_rows"] == 32 and stats["rows_rescanned"] == 0, stats
    assert_parity(p, got)


@pytest.mark.parametrize("max_ctas", [0, 16])
def test_fused_split_heaviest_blocks_first(mqa, max_ctas):
    """Eight requests of 8 rows with 64K, 8K and 4K keys: fewer blocks than
    CTAs and of very different lengths, so only the heaviest blocks are cut
    into key chunks (6 blocks x 16 chunks on every SM, 2 x 4 on 16 CTAs), and
    their chunks are claimed before the whole blocks.  Exact top-k."""
    p = synth.make_multi("split_first", (65536, 65536, 8192, 8192, 8192, 8192, 4096, 4096), (8,) * 8, 512, seed=3)
    debug = {"max_ctas": max_ctas} if max_ctas else None
    got, status, stats = run_fused(mqa, p, debug=debug)
    assert status == 0, stats
    assert 0 < stats["split_blocks"] < 8, stats
    assert stats["rows_rescanned"] == 0, stats
    assert_parity(p, got)


@pytest.mark.parametrize("seed,rows,keys,topk", [(40, 3, 700, 512), (41, 13, 5000, 1024), (42, 37, 20000, 2048)])
def test_fused_64_heads_random_ranges(mqa, seed, rows, keys, topk):
    """64 index heads per row (4-row blocks): arbitrary ranges, exact top-k."""
    p = synth.random_small(seed, rows, keys, topk, heads=64)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert_parity(p, got)


def test_fused_64_heads_gated_split(mqa):
    """64 index heads, long causal rows: sampled gate, binned selection and
    key chunks merged across CTAs."""
    p = _causal(synth.random_small(43, 16, 60000, 2048, heads=64, empty_frac=0.0), 60000)
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert stats["gated_rows"] == 16 and stats["split_blocks"] == 4, stats
    assert_parity(p, got)


def run_blocks(mqa, p, btopk, debug=None):
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows)
    out = mqa.mqa_block_topk_prefill(q, k, sc, w, s, e, btopk, workspace=ws, debug=debug)
    status, stats = mqa.get_status(ws)
    return out.cpu().numpy(), status, stats


def assert_block_parity(p, got, btopk):
    rows = np.arange(p.rows)
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_block_rows(got, p, rows, scores, btopk)
    assert not bad, bad[:10]


@pytest.mark.parametrize("seed,rows,keys,btopk", [(50, 5, 900, 512), (51, 19, 9000, 512), (52, 33, 30000, 1024)])
def test_block_selection_random_ranges(mqa, seed, rows, keys, btopk):
    """Top blocks of 8 keys by their largest score, arbitrary ranges."""
    p = synth.random_small(seed, rows, keys, 512)
    got, status, stats = run_blocks(mqa, p, btopk)
    assert status == 0, stats
    assert_block_parity(p, got, btopk)


def test_block_selection_gated_split(mqa):
    """Long causal rows: the gate samples block scores, key chunks of a split
    block are merged, the top 2048 blocks are exact up to ties."""
    p = _causal(synth.random_small(53, 16, 200000, 2048, empty_frac=0.0), 200000)
    got, status, stats = run_blocks(mqa, p, 2048)
    assert status == 0, stats
    assert stats["gated_rows"] == 16 and stats["rows_rescanned"] == 0, stats
    assert_block_parity(p, got, 2048)


def test_block_selection_forced_rescan(mqa):
    """Gate forced to +inf: every row under-fills and is rescanned exactly."""
    p = synth.random_small(54, 12, 40000, 512, empty_frac=0.0)
    got, status, stats = run_blocks(mqa, p, 512, debug={"force_gate": 1})
    assert status == 0, stats
    assert stats["rows_rescanned"] > 0
    assert_block_parity(p, got, 512)


def run_masked(mqa, p, mask, items, debug=None):
    import torch
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows)
    m = torch.from_numpy(mask.view(np.int32)).cuda()
    it = torch.from_numpy(items).cuda()
    out = mqa.mqa_topk_prefill_masked(q, k, sc, w, s, e, m, it, p.topk, workspace=ws, debug=debug)
    status, stats = mqa.get_status(ws)
    return out.cpu().numpy(), status, stats


def assert_masked_parity(p, got, mask):
    rows = np.arange(p.rows)
    _, scores = oracle.run_masked(p, mask, rows=rows, want_topk=False, want_scores=True)
    bad = check_masked_rows(got, p, rows, scores)
    assert not bad, bad[:10]


def test_block_mask_kernel_bit_exact(mqa):
    """The list-to-mask kernel equals the CPU construction, counts included."""
    import torch
    rng = np.random.default_rng(70)
    rows, keys, L = 40, 70000, 300
    starts = rng.integers(0, keys, rows).astype(np.int32)
    ends = np.minimum(keys, starts + rng.integers(0, 30000, rows)).astype(np.int32)
    lists = rng.integers(-1, 4000, (rows, L)).astype(np.int32)
    words = ((keys + 1023) // 1024) * 4
    want_m, want_i = numpy_block_mask(lists, starts, ends, keys, words)
    t = lambda a: torch.from_numpy(a).cuda()
    m, it = mqa.block_mask(t(lists), t(starts), t(ends), keys, words)
    assert np.array_equal(m.cpu().numpy().view(np.uint32), want_m)
    assert np.array_equal(it.cpu().numpy(), want_i)


@pytest.mark.parametrize("scan", [0, 1], ids=["gather", "scan"])
@pytest.mark.parametrize("seed,rows,keys,topk,frac", [(71, 9, 3000, 512, 0.5), (72, 24, 40000, 512, 0.3),
                                                      (73, 17, 90000, 1024, 0.05), (76, 13, 120000, 2048, 0.6)])
def test_masked_selection_random_masks(mqa, seed, rows, keys, topk, frac, scan):
    """Top-k over the keys of each row's allowed blocks (random masks), by
    the gathering kernel (rows of up to ~2,400 allowed blocks: up to four
    768-block jobs and a running top-k) and by the masked scan."""
    p = synth.random_small(seed, rows, keys, topk)
    rng = np.random.default_rng(seed)
    picks = rng.integers(0, keys // 8 + 1, (rows, 4096))  # relative block indices, many past the range
    lists = np.where(rng.random((rows, 4096)) < frac, picks, -1).astype(np.int32)
    words = ((keys + 1023) // 1024) * 4
    mask, items = numpy_block_mask(lists, p.starts, p.ends, keys, words)
    got, status, stats = run_masked(mqa, p, mask, items, debug={"masked_scan": scan})
    assert status == 0, stats
    if scan == 0:
        assert stats["blocks_done"] == rows and stats["candidates"] == int(items.sum()), stats
    assert_masked_parity(p, got, mask)


def _full_mask(p):
    words = ((p.keys + 1023) // 1024) * 4
    mask = np.full((p.rows, words), 0xFFFFFFFF, np.uint32)
    items = np.maximum(p.ends - p.starts, 0).astype(np.int32)
    return mask, items


def test_masked_gather_full_mask_equals_unmasked(mqa):
    """A mask that allows every block: the gathering kernel's selection is the
    unmasked top-k (rows of up to 6,250 blocks, nine jobs each)."""
    p = synth.random_small(77, 20, 50000, 512)
    mask, items = _full_mask(p)
    got, status, stats = run_masked(mqa, p, mask, items)
    assert status == 0, stats
    assert stats["candidates"] == int(items.sum()), stats
    assert_parity(p, got)


def test_masked_gather_job_boundaries(mqa):
    """Rows whose allowed blocks number exactly 768 (one full job), 769 (a
    second job of one block), 1,536, 2,304 (three full jobs: every job slot
    in use for one row), 1,024, 3,000, one, none, and blocks cut by the range
    at both ends; one CTA serves every row, reusing each job slot."""
    rng = np.random.default_rng(78)
    keys, rows = 60000, 11
    p = synth.random_small(78, rows, keys, 512, empty_frac=0.0)
    starts = np.array([3, 1001, 5, 17, 0, 999, 100, 50003, 8, 2, 640], np.int32)
    ends = np.array([59997, 41005, 30000, 59999, 60000, 999, 9000, 50013, 59000, 52001, 60000], np.int32)
    p = synth.Problem(p.name, p.q, p.k, p.scales_ue8m0, p.weights, starts, ends, 512)
    words = ((keys + 1023) // 1024) * 4
    mask = np.zeros((rows, words), np.uint32)

    def allow(r, blocks):
        for b in blocks:
            mask[r, b // 32] |= np.uint32(1 << (b % 32))
    for r, nb in ((0, 768), (1, 769), (2, 1536), (4, 3000), (8, 2304), (9, 1024), (10, 2305)):
        lo, hi = int(starts[r]) // 8, (int(ends[r]) - 1) // 8
        allow(r, rng.choice(np.arange(lo, hi + 1), size=nb, replace=False))
    allow(3, [17 // 8])                          # one block, cut by the start
    allow(6, [100 // 8, (9000 - 1) // 8, 500])   # both end blocks cut by the range
    allow(7, [50003 // 8, 50012 // 8])           # a 10-key row
    mask[5, :] = 0xFFFFFFFF                      # an empty range
    _, items = _full_mask(p)
    got, status, stats = run_masked(mqa, p, mask, items, debug={"max_ctas": 1})
    assert status == 0, stats
    assert stats["blocks_done"] == rows, stats
    assert_masked_parity(p, got, mask)


def test_masked_gather_ties(mqa):
    """Every key identical (one k row, one scale): each row's scores are all
    equal, so the selection's value range is degenerate and it takes the
    full radix select; half the keys identical in a second case, so the
    threshold bin holds thousands of ties (more than the copy holds)."""
    base = synth.random_small(94, 12, 20000, 512, empty_frac=0.0)
    for frac in (1.0, 0.5):
        k = base.k.copy()
        g = base.scales_ue8m0.copy()
        n = int(frac * base.keys)
        k[:n] = k[0]
        g[:n] = g[0]
        p = synth.Problem(base.name, base.q, k, g, base.weights, base.starts, base.ends, base.topk)
        mask, items = _full_mask(p)
        got, status, stats = run_masked(mqa, p, mask, items)
        assert status == 0, stats
        assert_parity(p, got)


def test_masked_gather_timeout_then_recovers(mqa):
    """A stalled gathering kernel ends at the time limit with the timeout bit;
    the next call on the same context is correct."""
    p = synth.random_small(79, 12, 20000, 512)
    mask, items = _full_mask(p)
    _, status, _ = run_masked(mqa, p, mask, items, debug={"stall": 1, "wait_timeout_ms": 200})
    assert status & 2
    got, status, stats = run_masked(mqa, p, mask, items)
    assert status == 0, stats
    assert_parity(p, got)


def _expected_skipped_tiles(p, mask, block_rows=8):
    """Main tiles of each row block's key range (the union of its rows'
    ranges) in which no row of the block allows a key."""
    total = 0
    for b0 in range(0, p.rows, block_rows):
        rr = [r for r in range(b0, min(p.rows, b0 + block_rows)) if p.ends[r] > p.starts[r]]
        if not rr:
            continue
        lo = min(int(p.starts[r]) for r in rr)
        hi = max(int(p.ends[r]) for r in rr)
        for t in range(lo // 128, (hi + 127) // 128):
            half = (mask[b0:b0 + block_rows, t // 2] >> np.uint32(16 * (t % 2))) & np.uint32(0xFFFF)
            total += int(not half.any())
    return total


def test_masked_skips_tiles_without_allowed_keys(mqa):
    """The masked scan: each row allows blocks in one narrow window of a long
    range; the tiles no row of a block allows are left out (counted exactly
    when no row is rescanned) and the result still equals the oracle's."""
    rng = np.random.default_rng(75)
    p = synth.random_small(75, 24, 200000, 512, empty_frac=0.0)
    keys = p.keys
    lists = np.full((p.rows, 1024), -1, np.int32)
    for r in range(p.rows):
        nb = (int(p.ends[r]) - 1) // 8 - int(p.starts[r]) // 8 + 1
        win = min(nb, 2000)
        w0 = int(rng.integers(0, nb - win + 1))
        pick = w0 + rng.choice(win, size=min(700, win), replace=False)
        lists[r, :len(pick)] = pick
    words = ((keys + 1023) // 1024) * 4
    mask, items = numpy_block_mask(lists, p.starts, p.ends, keys, words)
    got, status, stats = run_masked(mqa, p, mask, items, debug={"masked_scan": 1})
    assert status == 0, stats
    want = _expected_skipped_tiles(p, mask)
    assert want > 0
    if stats["rows_rescanned"] == 0:
        assert stats["skipped_tiles"] == want, (stats, want)
    else:
        assert stats["skipped_tiles"] >= want, (stats, want)
    assert_masked_parity(p, got, mask)


def test_two_level_source_then_consumer(mqa):
    """The two-level chain on long causal rows: the oracle's top 2048 blocks of
    8 keys (source) restrict the consumer's top-512."""
    p = _causal(synth.random_small(74, 16, 200000, 512, empty_frac=0.0), 200000)
    lists = oracle.run_blocks(p, 2048)
    words = ((p.keys + 1023) // 1024) * 4
    mask, items = numpy_block_mask(lists, p.starts, p.ends, p.keys, words)
    got, status, stats = run_masked(mqa, p, mask, items)
    assert status == 0, stats
    assert stats["blocks_done"] == 16 and stats["candidates"] == int(items.sum()), stats
    assert_masked_parity(p, got, mask)
    got, status, stats = run_masked(mqa, p, mask, items, debug={"masked_scan": 1})
    assert status == 0, stats
    assert stats["gated_rows"] == 16, stats
    assert_masked_parity(p, got, mask)


def test_host_buffer_entry(mqa):
    """mqa_topk_prefill_host: host inputs in, host indices out, through the C
    ABI on one stream; two calls in a row on one staging buffer."""
    import torch
    for seed in (90, 91):
        p = synth.random_small(seed, 40, 30000, 512)
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        staging = mqa.alloc_host_staging(p.rows, p.keys, p.topk)
        out = torch.full((p.rows, p.topk), 7, dtype=torch.int32).pin_memory()
        s = torch.cuda.Stream()
        mqa.mqa_topk_prefill_host(pin(p.q), pin(p.k), pin(p.scales_ue8m0), pin(p.weights), pin(p.starts),
                                  pin(p.ends), p.topk, staging, out, stream=s)
        s.synchronize()
        status, stats = mqa.host_get_status(staging, p.rows, p.keys, p.topk)
        assert status == 0, stats
        assert_parity(p, out.numpy())


def test_fused_single_cta(mqa):
    """All blocks through one persistent CTA (job slots and slabs reused many times)."""
    p = synth.random_small(23, 64, 9000, 512)
    got, status, stats = run_fused(mqa, p, debug={"max_ctas": 1})
    assert status == 0, stats
    assert_parity(p, got)


def test_workspace_reuse_two_calls(mqa):
    p = synth.random_small(24, 20, 7000, 512)
    ws = mqa.alloc_workspace(p.rows)
    a, s1, _ = run_fused(mqa, p, workspace=ws)
    b, s2, _ = run_fused(mqa, p, workspace=ws)
    assert s1 == 0 and s2 == 0
    assert_parity(p, a)
    assert_parity(p, b)


def test_bounded_wait_reports_timeout(mqa):
    """A wait that nothing completes ends at the time limit with a status bit;
    the context stays usable for the next call."""
    p = synth.random_small(25, 8, 1000, 512)
    _, status, _ = run_fused(mqa, p, debug={"stall": 1, "wait_timeout_ms": 200})
    assert status & 2
    got, status, _ = run_fused(mqa, p)
    assert status == 0
    assert_parity(p, got)


def test_fused_max_keys(mqa):
    """2^24 keys, the largest key count the library accepts (K is 2 GiB):
    ranges that end at the last key, one gated 400K-key range, one at key 0.
    Each row is checked against the oracle on its own key window."""
    p = synth.max_keys()
    got, status, stats = run_fused(mqa, p)
    assert status == 0, stats
    assert stats["gated_rows"] >= 1, stats
    for r in range(p.rows):
        sub = synth.window(p, r)
        _, scores = oracle.run(sub, want_topk=False, want_scores=True)
        bad = check_topk_rows(got[r:r + 1], sub, np.array([0]), scores)
        assert not bad, (r, bad[:5])


def test_masked_gather_max_keys(mqa):
    """The gathering kernel at 2^24 keys (K is 2 GiB): each row allows up to
    3,000 random blocks of its range (ranges ending at the last key, one at
    key 0, unaligned starts); every row is checked against the oracle on a
    block-aligned window of its keys."""
    p = synth.max_keys(topk=512)
    keys = p.keys
    rng = np.random.default_rng(93)
    nb = ((p.ends.astype(np.int64) - 1) // 8 - p.starts.astype(np.int64) // 8 + 1).clip(min=1)
    lists = np.full((p.rows, 3000), -1, np.int32)
    for r in range(p.rows):
        pick = rng.choice(int(nb[r]), size=min(3000, int(nb[r])), replace=False)
        lists[r, :len(pick)] = pick
    words = ((keys + 1023) // 1024) * 4
    mask, items = numpy_block_mask(lists, p.starts, p.ends, keys, words)
    got, status, stats = run_masked(mqa, p, mask, items)
    assert status == 0, stats
    assert stats["blocks_done"] == p.rows and stats["candidates"] == int(items.sum()), stats
    for r in range(p.rows):
        s, e = int(p.starts[r]), int(p.ends[r])
        s8 = s - s % 8
        sub = synth.Problem(f"{p.name}_w{r}", p.q[r:r + 1], p.k[s8:e], p.scales_ue8m0[s8:e], p.weights[r:r + 1],
                            np.array([s - s8], np.int32), np.array([e - s8], np.int32), p.topk)
        wk = e - s8
        wwords = ((wk + 1023) // 1024) * 4
        wmask = np.zeros((1, wwords), np.uint32)
        b0 = s8 // 8
        for b in range((wk + 7) // 8):
            if (mask[r, (b0 + b) // 32] >> np.uint32((b0 + b) % 32)) & np.uint32(1):
                wmask[0, b // 32] |= np.uint32(1 << (b % 32))
        _, scores = oracle.run_masked(sub, wmask, want_topk=False, want_scores=True)
        bad = check_masked_rows(got[r:r + 1], sub, np.array([0]), scores)
        assert not bad, (r, bad[:5])


def test_fused_cuda_graph_replay(mqa):
    """The fused call captured into a CUDA graph (one memset node and one
    kernel node on the caller's workspace) and replayed: every replay gives
    the exact top-k, also after the inputs change in place."""
    import torch
    p = synth.random_small(28, 40, 30000, 1024, empty_frac=0.05)
    q, k, sc, w, s, e = to_device(p)
    ws = mqa.alloc_workspace(p.rows)
    out = torch.empty((p.rows, p.topk), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk, workspace=ws, out=out)  # first use outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk, workspace=ws, out=out)
    for _ in range(3):
        out.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        status, stats = mqa.get_status(ws)
        assert status == 0, stats
        assert_parity(p, out.cpu().numpy())
    # new weights in place: the replay reads the current inputs
    p2 = synth.random_small(29, 40, 30000, 1024, empty_frac=0.05)
    p2.q, p2.k, p2.scales_ue8m0, p2.starts, p2.ends = p.q, p.k, p.scales_ue8m0, p.starts, p.ends
    w.copy_(torch.from_numpy(p2.weights).cuda())
    g.replay()
    torch.cuda.synchronize()
    assert_parity(p2, out.cpu().numpy())


@pytest.mark.parametrize("name", ["random", "r2048_32k_k512"])
def test_fold_prep_bit_exact(mqa, name):
    """Folded query terms: codes and exponents bit for bit against the oracle
    (both decide them in fp32), the residual norm to fp32 rounding; rows with
    weights scaled by 1e6 and 1e-6 and an all-zero row included."""
    import torch
    if name == "random":
        p = synth.random_small(96, 37, 10, 512)
        p.weights[3] *= 1e6
        p.weights[4] *= 1e-6
        p.weights[5] = 0.0
    else:
        p = synth.make(name)
    q = torch.from_numpy(p.q).cuda()
    w = torch.from_numpy(p.weights).cuda()
    codes, exps, beta = mqa.fold_prep(q, w)
    oc, oe, _, ob = oracle.fold_prep(p.q, p.weights)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(exps.cpu().numpy(), oe)
    assert np.allclose(beta.cpu().numpy().astype(np.float64), ob, rtol=1e-5, atol=0.0)


def test_out_of_range_rows_clamped(mqa):
    p = synth.random_small(26, 8, 3000, 512)
    p.starts[0], p.ends[0] = -5, 700
    p.starts[1], p.ends[1] = 2900, 3400
    got, status, _ = run_fused(mqa, p)
    assert status & 1
    # the oracle rejects such rows; compare against the clamped problem
    p.starts[0], p.ends[0] = 0, 700
    p.starts[1], p.ends[1] = 2900, 3000
    # indices are relative to the clamped start
    assert_parity(p, got)


# ---------------------------------------------------------------- dense baseline
@pytest.mark.parametrize("budget_rows", [1000, 7, 1])
def test_dense_baseline(mqa, budget_rows):
    p = synth.random_small(30, 20, 6000, 512)
    q, k, sc, w, s, e = to_device(p)
    out = mqa.mqa_topk_dense_baseline(q, k, sc, w, s, e, p.topk, logits_budget_bytes=budget_rows * p.keys * 4)
    assert_parity(p, out.cpu().numpy())


def test_dense_matches_fused_tiny(mqa):
    p = synth.make("tiny_64x4096_k512")
    q, k, sc, w, s, e = to_device(p)
    out = mqa.mqa_topk_dense_baseline(q, k, sc, w, s, e, p.topk).cpu().numpy()
    assert_parity(p, out)
