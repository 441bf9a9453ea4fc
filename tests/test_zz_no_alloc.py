"""The allocation-free entry point `mqa_topk_prefill_noalloc`.

It serves callers that cannot allocate device memory (a stream being captured
into a CUDA graph in global capture mode, where cudaMalloc is not permitted; a
plugin whose host framework owns the device memory pool).  Instead of a
caller-provided workspace it uses a fixed static device array inside the
library.  Its output must match the workspace entry point's under the same
tie rule as every other parity test, on two calls in a row (the scratch keeps
the previous call's contents, so the second call checks that the state that
must start at zero is cleared).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from parity import TOPK_TIE_TOL, to_device

pytestmark = pytest.mark.gpu


def same_up_to_ties(a, b, p, scores):
    for i in range(p.rows):
        s, e = int(p.starts[i]), int(p.ends[i])
        n = max(0, e - s)
        c = min(p.topk, n)
        assert np.all(a[i, c:] == -1) and np.all(b[i, c:] == -1)
        sa, sb = set(a[i, :c].tolist()), set(b[i, :c].tolist())
        assert len(sa) == c and len(sb) == c
        if sa == sb:
            continue
        vis = scores[i, s:e]
        kth = np.sort(vis)[::-1][c - 1]
        tol = TOPK_TIE_TOL * np.max(np.abs(vis))
        for j in sa ^ sb:
            assert abs(vis[j] - kth) <= tol, (i, j)


@pytest.mark.parametrize("maker", [lambda: synth.make("tiny_64x4096_k512"),
                                   lambda: synth.random_small(41, 40, 30000, 1024, empty_frac=0.05)])
def test_noalloc_matches_workspace_entry_twice(maker):
    import torch
    import sparse_attention_indexer_relu_gb300 as mqa
    assert torch.cuda.is_available()
    p = maker()
    q, k, sc, w, s, e = to_device(p)
    ref = mqa.mqa_topk_prefill(q, k, sc, w, s, e, p.topk).cpu().numpy()
    _, scores = oracle.run(p, want_topk=False, want_scores=True)
    L = mqa.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    for call in range(2):
        out = torch.full((p.rows, p.topk), 7, dtype=torch.int32, device="cuda")
        rc = L.mqa_topk_prefill_noalloc(P(q), P(k), P(sc), P(w), P(s), P(e), P(out), p.rows, p.keys, p.topk,
                                        stream)
        assert rc == 0, mqa.strerror(rc)
        torch.cuda.synchronize()
        same_up_to_ties(out.cpu().numpy(), ref, p, scores)
