"""The allocation-free entry point `mqa_topk_prefill_noalloc`.

It serves callers that cannot allocate device memory: code that runs while a
stream is being captured into a CUDA graph in global capture mode (cudaMalloc
is not permitted there), and plugins whose host framework owns the device
memory pool.  Instead of a caller-provided workspace it uses a fixed static
device array inside the library, which keeps the previous call's contents.
Each case runs two calls in a row on DIFFERENT inputs (other rows, keys,
top-k and block counts), so a second call could only pass with stale scratch
if its reset of the state that must start at zero were missing; both results
are checked against the oracle under the pass rule of every parity test, and
the device status is read through `mqa_topk_noalloc_get_status`.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from parity import check_topk_rows, to_device

pytestmark = pytest.mark.gpu


def noalloc(mqa, p):
    import torch
    q, k, sc, w, s, e = to_device(p)
    L = mqa.lib()
    out = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.mqa_topk_prefill_noalloc(P(q), P(k), P(sc), P(w), P(s), P(e), P(out), p.rows, p.keys, p.topk, stream)
    assert rc == 0, mqa.strerror(rc)
    status, stats = mqa.noalloc_get_status()
    return out.cpu().numpy(), status, stats


def assert_oracle(p, got):
    rows = np.arange(p.rows)
    _, scores = oracle.run(p, rows=rows, want_topk=False, want_scores=True)
    bad = check_topk_rows(got, p, rows, scores)
    assert not bad, bad[:10]


def causal(p):
    p.starts = np.zeros(p.rows, np.int32)
    p.ends = (p.keys - p.rows + 1 + np.arange(p.rows)).astype(np.int32)
    return p


PAIRS = {
    # many blocks on at most 8 CTAs, then a small chunk with empty rows
    "tiny_then_random": (lambda: synth.make("tiny_64x4096_k512"),
                         lambda: synth.random_small(41, 40, 30000, 1024, empty_frac=0.05)),
    # one 8-row block whose gated rows are split into key chunks, then a
    # different single block with another top-k
    "one_block_twice": (lambda: causal(synth.random_small(42, 8, 60000, 2048, empty_frac=0.0)),
                        lambda: causal(synth.random_small(43, 5, 20000, 512, empty_frac=0.0))),
}


@pytest.mark.parametrize("name", sorted(PAIRS))
def test_noalloc_two_different_calls_match_oracle(name):
    import torch
    import sparse_attention_indexer_relu_gb300 as mqa
    assert torch.cuda.is_available()
    first, second = PAIRS[name]
    for make in (first, second):
        p = make()
        got, status, stats = noalloc(mqa, p)
        assert status == 0, stats
        assert stats["blocks_done"] >= (p.rows + 7) // 8, stats
        assert_oracle(p, got)
