"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before any device work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_relu_gb300 as mqa

HEADER = mqa.HEADER_PATH


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mqa_[a-z0-9_]+)\s*\(", text)))


def test_library_builds_and_loads():
    from sparse_attention_indexer_relu_gb300 import build
    build.build()
    assert os.path.exists(mqa.LIB_PATH)
    mqa.lib()


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(mqa.EXPORTS), names
    L = ctypes.CDLL(mqa.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_strerror_codes():
    assert mqa.strerror(0) == "ok"
    for code in range(1, 7):
        assert mqa.strerror(code) not in ("ok", "unknown error")
    assert mqa.strerror(99) == "unknown error"


P = ctypes.c_void_p


def call_prefill(rows=8, keys=100, topk=512, q=0x1000, k=0x2000, sc=0x3000, w=0x4000, s=0x5000, e=0x6000,
                 out=0x7000, ws=0x100000, ws_bytes=1 << 30):
    return mqa.lib().mqa_topk_prefill(P(q), P(k), P(sc), P(w), P(s), P(e), P(out), rows, keys, topk, P(ws),
                                      ws_bytes, None)


# argument errors are found before any CUDA call, so fake device addresses are safe here
def test_prefill_rejects_bad_topk():
    for t in (0, 1, 100, 511, 4096):
        assert call_prefill(topk=t) == 1


def test_prefill_rejects_bad_sizes():
    assert call_prefill(rows=-1) == 1
    assert call_prefill(keys=0) == 1
    assert call_prefill(keys=(1 << 24) + 1) == 1


def test_prefill_rejects_null_and_misaligned():
    assert call_prefill(q=0) == 1
    assert call_prefill(out=0) == 1
    assert call_prefill(ws=0) == 1
    assert call_prefill(q=0x1001) == 2
    assert call_prefill(k=0x2008) == 2
    assert call_prefill(sc=0x3004) == 2
    assert call_prefill(out=0x7004) == 2
    assert call_prefill(s=0x5002) == 2
    assert call_prefill(ws=0x100010) == 2


def test_prefill_zero_rows_is_noop():
    assert call_prefill(rows=0) == 0


def test_debug_options_validated():
    opt = mqa.DebugOptions(force_gate=3)
    rc = mqa.lib().mqa_topk_prefill_debug(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), P(0x6000),
                                          P(0x7000), 8, 100, 512, P(0x100000), 1 << 30, None, ctypes.byref(opt))
    assert rc == 1
    opt = mqa.DebugOptions(slab_capacity=600)  # below topk + 256
    rc = mqa.lib().mqa_topk_prefill_debug(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), P(0x6000),
                                          P(0x7000), 8, 100, 512, P(0x100000), 1 << 30, None, ctypes.byref(opt))
    assert rc == 1


def test_ue8m0_argument_checks():
    L = mqa.lib()
    assert L.mqa_ue8m0_decode(P(0x1000), P(0x2000), -1, None) == 1
    assert L.mqa_ue8m0_decode(None, None, 0, None) == 0
    assert L.mqa_ue8m0_decode(None, P(0x2000), 5, None) == 1
    assert L.mqa_ue8m0_decode(P(0x1001), P(0x2000), 5, None) == 2


def test_host_entry_argument_checks():
    """Argument errors of the host-buffer entry come back before any device
    work (no GPU needed)."""
    L = mqa.lib()
    h = [P(0x1000 * i) for i in range(1, 8)]
    # bad sizes and topk
    assert L.mqa_topk_prefill_host(*h, 8, 0, 512, P(0x100000), 1 << 30, None) == 1
    assert L.mqa_topk_prefill_host(*h, -1, 100, 512, P(0x100000), 1 << 30, None) == 1
    assert L.mqa_topk_prefill_host(*h, 8, 100, 300, P(0x100000), 1 << 30, None) == 1
    # zero rows is a no-op; null buffers and a misaligned staging buffer are rejected
    assert L.mqa_topk_prefill_host(*h, 0, 100, 512, P(0x100000), 1 << 30, None) == 0
    assert L.mqa_topk_prefill_host(None, *h[1:], 8, 100, 512, P(0x100000), 1 << 30, None) == 1
    assert L.mqa_topk_prefill_host(*h, 8, 100, 512, None, 1 << 30, None) == 1
    assert L.mqa_topk_prefill_host(*h, 8, 100, 512, P(0x100010), 1 << 30, None) == 2
    n = ctypes.c_size_t()
    assert L.mqa_topk_host_staging_bytes(0, 8, 100, 300, ctypes.byref(n)) == 1
    assert L.mqa_topk_host_get_status(None, 8, 100, 512, None, None, None) == 1


def test_logits_and_dense_argument_checks():
    L = mqa.lib()
    args = [P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), P(0x6000), P(0x7000), 8, 100]
    assert L.mqa_logits_debug(*args, P(0x100000), 16, None) == 3   # header too small
    assert L.mqa_logits_debug(*args, P(0x100008), 256, None) == 2  # misaligned header
    assert L.mqa_topk_dense_baseline(*args, 512, P(0x8000), 399, P(0x100000), 256, None) == 3  # < one row
    assert L.mqa_topk_dense_baseline(*args, 100, P(0x8000), 1 << 20, P(0x100000), 256, None) == 1


def test_status_argument_checks():
    assert mqa.lib().mqa_topk_get_status(None, None, None, None) == 1


def test_workspace_query_without_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present")
    n = ctypes.c_size_t(0)
    assert mqa.lib().mqa_topk_workspace_bytes(0, 16, ctypes.byref(n)) in (5, 6)


def test_fold_prep_rejects_bad_arguments():
    L = mqa.lib()
    assert L.mqa_fold_prep(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), -1, None) == 1
    assert L.mqa_fold_prep(P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 0, None) == 0
    assert L.mqa_fold_prep(None, P(0x2000), P(0x3000), P(0x4000), P(0x5000), 4, None) == 1
    assert L.mqa_fold_prep(P(0x1001), P(0x2000), P(0x3000), P(0x4000), P(0x5000), 4, None) == 2
    assert L.mqa_fold_prep(P(0x1000), P(0x2000), P(0x3008), P(0x4000), P(0x5000), 4, None) == 2
