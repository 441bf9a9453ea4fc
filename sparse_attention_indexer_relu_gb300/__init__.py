"""Fused FP8 MQA-logits + per-row top-k selection for GB300 (sm_103a).

Thin Python binding over the C ABI in `include/mqatopk.h` (library
`_build/libmqatopk.so`, built by `build.py`).  It only marshals arguments:
torch provides device memory and streams, every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or the device is not supported, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import plan  # noqa: F401  (host-side sizing rules)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmqatopk.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "mqatopk.h")

HEADS = 32
HEAD_DIM = 128
TOPKS = (512, 1024, 2048)
HEADER_BYTES = 256
DEFAULT_SLAB_CAP = 13312
DEFAULT_LOGITS_BUDGET = 512 * 2 ** 20

MQA_OK = 0
STATUS_BITS = {1: "range_clamped", 2: "wait_timeout", 4: "internal"}
STAT_NAMES = ("status", "rows_rescanned", "compactions", "candidates", "gated_rows", "blocks_done",
              "sample_tiles", "overflow_rows", "underfill_rows", "select_fallback",
              "kernel_us", "end_spread_us", "split_blocks", "unsafe_rows", "fold_bound_ppm", "pair_rows",
              "skipped_tiles")

EXPORTS = ("mqa_topk_workspace_bytes", "mqa_topk_workspace_bytes_ex", "mqa_topk_prefill", "mqa_topk_prefill_ex",
           "mqa_block_topk_prefill", "mqa_topk_prefill_masked", "mqa_block_mask",
           "mqa_topk_prefill_debug", "mqa_topk_prefill_noalloc", "mqa_topk_noalloc_get_status",
           "mqa_ue8m0_decode", "mqa_fold_prep", "mqa_logits_debug", "mqa_topk_dense_baseline", "mqa_topk_get_status",
           "mqa_fp8_mma_probe", "mqa_topk_host_staging_bytes", "mqa_topk_prefill_host", "mqa_topk_host_get_status",
           "mqa_topk_strerror")


class MQAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


class DebugOptions(ctypes.Structure):
    _fields_ = [("force_gate", ctypes.c_int), ("slab_capacity", ctypes.c_int), ("stall", ctypes.c_int),
                ("wait_timeout_ms", ctypes.c_int), ("max_ctas", ctypes.c_int), ("force_unsafe", ctypes.c_int),
                ("head_sum", ctypes.c_int), ("masked_scan", ctypes.c_int)]


_lib = None


def lib():
    """The loaded C library (ctypes), argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmqatopk.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.mqa_topk_workspace_bytes.argtypes = [I, I, ctypes.POINTER(S)]
    L.mqa_topk_workspace_bytes_ex.argtypes = [I, I, I, ctypes.POINTER(S)]
    common = [P, P, P, P, P, P, P, I, I]
    L.mqa_topk_prefill.argtypes = common + [I, P, S, P]
    L.mqa_topk_prefill_debug.argtypes = common + [I, P, S, P, ctypes.POINTER(DebugOptions)]
    L.mqa_topk_prefill_ex.argtypes = common + [I, I, P, S, P, ctypes.POINTER(DebugOptions)]
    L.mqa_block_topk_prefill.argtypes = common + [I, P, S, P, ctypes.POINTER(DebugOptions)]
    L.mqa_topk_prefill_masked.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I, I, P, S, P, ctypes.POINTER(DebugOptions)]
    L.mqa_block_mask.argtypes = [P, P, P, I, I, I, P, I, P, P]
    L.mqa_topk_prefill_noalloc.argtypes = common + [I, P]
    L.mqa_topk_noalloc_get_status.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), P]
    L.mqa_ue8m0_decode.argtypes = [P, P, I, P]
    L.mqa_fp8_mma_probe.argtypes = [ctypes.c_longlong, P, P]
    L.mqa_topk_host_staging_bytes.argtypes = [I, I, I, I, ctypes.POINTER(S)]
    L.mqa_topk_prefill_host.argtypes = [P, P, P, P, P, P, P, I, I, I, P, S, P]
    L.mqa_topk_host_get_status.argtypes = [P, I, I, I, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), P]
    L.mqa_fold_prep.argtypes = [P, P, P, P, P, I, P]
    L.mqa_logits_debug.argtypes = common + [P, S, P]
    L.mqa_topk_dense_baseline.argtypes = common + [I, P, S, P, S, P]
    L.mqa_topk_get_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), P]
    L.mqa_topk_strerror.argtypes = [I]
    L.mqa_topk_strerror.restype = ctypes.c_char_p
    for name in EXPORTS[:-1]:
        getattr(L, name).restype = I
    _lib = L
    return L


def strerror(code: int) -> str:
    return lib().mqa_topk_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != MQA_OK:
        raise MQAError(rc, what)


# ---------------------------------------------------------------- marshalling helpers
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _as_u8(t, shape, name):
    torch = _torch()
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must be uint8 e4m3fn codes or float8_e4m3fn, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def _as(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def _inputs(q, k, key_scales, weights, starts, ends, heads=(HEADS,)):
    torch = _torch()
    rows, keys = int(q.shape[0]), int(k.shape[0])
    h = int(q.shape[1]) if q.dim() == 3 and int(q.shape[1]) in heads else HEADS
    q = _as_u8(q, (rows, h, HEAD_DIM), "q")
    k = _as_u8(k, (keys, HEAD_DIM), "k")
    key_scales = _as(key_scales, torch.float32, (keys,), "key_scales")
    weights = _as(weights, torch.float32, (rows, h), "weights")
    starts = _as(starts, torch.int32, (rows,), "starts")
    ends = _as(ends, torch.int32, (rows,), "ends")
    return q, k, key_scales, weights, starts, ends, rows, keys


# ---------------------------------------------------------------- public API
def workspace_bytes(rows: int, device: Optional[int] = None, heads: int = HEADS) -> int:
    torch = _torch()
    dev = torch.cuda.current_device() if device is None else int(device)
    n = ctypes.c_size_t(0)
    _check(lib().mqa_topk_workspace_bytes_ex(dev, int(rows), int(heads), ctypes.byref(n)),
           "mqa_topk_workspace_bytes_ex")
    return int(n.value)


def alloc_workspace(rows: int, device=None, heads: int = HEADS):
    """One fixed-size workspace for calls over up to `rows` rows of `heads`
    index heads (caller owns it)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else int(device))
    return torch.empty(workspace_bytes(rows, dev.index, heads), dtype=torch.uint8, device=dev)


def ue8m0_decode(scales, out=None, stream=None):
    """[keys, 4] uint8 UE8M0 groups -> [keys] fp32 scales (bit pattern e << 23)."""
    torch = _torch()
    keys = int(scales.shape[0])
    scales = _as(scales, torch.uint8, (keys, 4), "scales")
    if out is None:
        out = torch.empty(keys, dtype=torch.float32, device=scales.device)
    _check(lib().mqa_ue8m0_decode(_ptr(scales), _ptr(out), keys, _stream(stream)), "mqa_ue8m0_decode")
    return out


def fp8_mma_probe(tiles_per_sm: int = 40000, device=None):
    """The tensor pipe's FP8 MMA ceiling in TFLOP/s: one timed launch of
    mqa_fp8_mma_probe (back-to-back 128 x 256 x 128 tiles on every SM) after
    a short warm-up launch."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    _check(lib().mqa_fp8_mma_probe(1000, _ptr(status), _stream(stream)), "mqa_fp8_mma_probe")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    _check(lib().mqa_fp8_mma_probe(int(tiles_per_sm), _ptr(status), _stream(stream)), "mqa_fp8_mma_probe")
    b.record(stream)
    b.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"fp8 probe status {int(status.item())}")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * tiles_per_sm * 2.0 * 128 * 256 * 128 / (a.elapsed_time(b) * 1e-3) / 1e12


FOLD_TERMS = 4


def fold_prep(q, weights, stream=None):
    """Folded query of each row as FOLD_TERMS e4m3 terms with power-of-two
    scales: returns (codes [rows, FOLD_TERMS, 128] uint8, exps [rows,
    FOLD_TERMS] int32, beta [rows] float32, the residual's 2-norm)."""
    torch = _torch()
    rows = int(q.shape[0])
    q = _as_u8(q, (rows, HEADS, 128), "q")
    weights = _as(weights, torch.float32, (rows, HEADS), "weights")
    codes = torch.empty((rows, FOLD_TERMS, 128), dtype=torch.uint8, device=q.device)
    exps = torch.empty((rows, FOLD_TERMS), dtype=torch.int32, device=q.device)
    beta = torch.empty(rows, dtype=torch.float32, device=q.device)
    _check(lib().mqa_fold_prep(_ptr(q), _ptr(weights), _ptr(codes), _ptr(exps), _ptr(beta), rows, _stream(stream)),
           "mqa_fold_prep")
    return codes, exps, beta


def mqa_topk_prefill(q, k, key_scales, weights, starts, ends, topk: int, workspace=None, out=None,
                     stream=None, debug: Optional[dict] = None):
    """Fused top-k prefill selection; returns out [rows, topk] int32 (relative
    indices, unordered, -1 padded).  q is [rows, 32 or 64, 128] (index heads
    taken from its shape), weights [rows, heads]."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends,
                                                                  heads=(32, 64))
    heads = int(q.shape[1])
    if out is None:
        out = torch.empty((rows, int(topk)), dtype=torch.int32, device=q.device)
    out = _as(out, torch.int32, (rows, int(topk)), "out")
    if workspace is None:
        workspace = alloc_workspace(rows, q.device.index, heads)
    args = [_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts), _ptr(ends), _ptr(out), rows, keys,
            int(topk), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)]
    if heads != HEADS:
        opt = DebugOptions(**{f: int((debug or {}).get(f, 0)) for f, _ in DebugOptions._fields_})
        _check(lib().mqa_topk_prefill_ex(*args[:10], heads, *args[10:], ctypes.byref(opt)), "mqa_topk_prefill_ex")
    elif debug:
        opt = DebugOptions(**{f: int(debug.get(f, 0)) for f, _ in DebugOptions._fields_})
        _check(lib().mqa_topk_prefill_debug(*args, ctypes.byref(opt)), "mqa_topk_prefill_debug")
    else:
        _check(lib().mqa_topk_prefill(*args), "mqa_topk_prefill")
    return out


def mqa_block_topk_prefill(q, k, key_scales, weights, starts, ends, btopk: int, workspace=None, out=None,
                           stream=None, debug: Optional[dict] = None):
    """Block selection: each row's btopk best blocks of 8 keys by their largest
    score, as block index - floor(start / 8); returns out [rows, btopk] int32
    (unordered, -1 padded)."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends)
    if out is None:
        out = torch.empty((rows, int(btopk)), dtype=torch.int32, device=q.device)
    out = _as(out, torch.int32, (rows, int(btopk)), "out")
    if workspace is None:
        workspace = alloc_workspace(rows, q.device.index)
    opt = DebugOptions(**{f: int((debug or {}).get(f, 0)) for f, _ in DebugOptions._fields_})
    _check(lib().mqa_block_topk_prefill(_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts), _ptr(ends),
                                        _ptr(out), rows, keys, int(btopk), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream),
                                        ctypes.byref(opt)), "mqa_block_topk_prefill")
    return out


def block_mask(block_lists, starts, ends, keys: int, mask_words: Optional[int] = None, stream=None):
    """Per-row block mask (and visible-key counts) from block lists [rows, L]
    int32 relative to floor(start / 8): returns (mask [rows, words] uint32,
    row_items [rows] int32)."""
    torch = _torch()
    rows, L = int(block_lists.shape[0]), int(block_lists.shape[1])
    words = mask_words or ((int(keys) + 1023) // 1024) * 4
    lists = _as(block_lists, torch.int32, (rows, L), "block_lists")
    mask = torch.empty((rows, words), dtype=torch.int32, device=lists.device)
    items = torch.empty(rows, dtype=torch.int32, device=lists.device)
    _check(lib().mqa_block_mask(_ptr(lists), _ptr(starts), _ptr(ends), rows, L, int(keys), _ptr(mask), words,
                                _ptr(items), _stream(stream)), "mqa_block_mask")
    return mask, items


def mqa_topk_prefill_masked(q, k, key_scales, weights, starts, ends, mask, row_items, topk: int, workspace=None,
                            out=None, stream=None, debug: Optional[dict] = None):
    """Top-k over the keys each row's block mask allows (see block_mask)."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends)
    if out is None:
        out = torch.empty((rows, int(topk)), dtype=torch.int32, device=q.device)
    out = _as(out, torch.int32, (rows, int(topk)), "out")
    if workspace is None:
        workspace = alloc_workspace(rows, q.device.index)
    opt = DebugOptions(**{f: int((debug or {}).get(f, 0)) for f, _ in DebugOptions._fields_})
    _check(lib().mqa_topk_prefill_masked(_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts),
                                         _ptr(ends), _ptr(mask), int(mask.shape[1]), _ptr(row_items), _ptr(out),
                                         rows, keys, int(topk), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream),
                                         ctypes.byref(opt)), "mqa_topk_prefill_masked")
    return out


def mqa_topk_prefill_noalloc(q, k, key_scales, weights, starts, ends, topk: int, out=None, stream=None):
    """Fused top-k without a workspace: the library uses its own fixed static
    device scratch (for callers that cannot allocate device memory).  Calls
    must not overlap on the GPU; the first call on a device must precede any
    stream capture."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends)
    if out is None:
        out = torch.empty((rows, int(topk)), dtype=torch.int32, device=q.device)
    out = _as(out, torch.int32, (rows, int(topk)), "out")
    _check(lib().mqa_topk_prefill_noalloc(_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts),
                                          _ptr(ends), _ptr(out), rows, keys, int(topk), _stream(stream)),
           "mqa_topk_prefill_noalloc")
    return out


def noalloc_get_status(stream=None):
    """(status bits, {counter name: value}) of the last mqa_topk_prefill_noalloc
    call on the current device (synchronises)."""
    st = ctypes.c_int32(0)
    stats = (ctypes.c_int32 * len(STAT_NAMES))()
    _check(lib().mqa_topk_noalloc_get_status(ctypes.byref(st), stats, _stream(stream)), "mqa_topk_noalloc_get_status")
    return int(st.value), dict(zip(STAT_NAMES, [int(v) for v in stats]))


def mqa_logits_debug(q, k, key_scales, weights, starts, ends, logits=None, workspace=None, stream=None):
    """[rows, keys] fp32 scores (-inf outside each row's range)."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends)
    if logits is None:
        logits = torch.empty((rows, keys), dtype=torch.float32, device=q.device)
    logits = _as(logits, torch.float32, (rows, keys), "logits")
    if workspace is None:
        workspace = torch.zeros(HEADER_BYTES, dtype=torch.uint8, device=q.device)
    _check(lib().mqa_logits_debug(_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts), _ptr(ends),
                                  _ptr(logits), rows, keys, _ptr(workspace), workspace.numel(), _stream(stream)),
           "mqa_logits_debug")
    return logits


def mqa_topk_dense_baseline(q, k, key_scales, weights, starts, ends, topk: int,
                            logits_budget_bytes: int = DEFAULT_LOGITS_BUDGET, logits_ws=None, workspace=None,
                            out=None, stream=None):
    """Dense comparison path: chunked fp32 logits, then per-row top-k."""
    torch = _torch()
    q, k, key_scales, weights, starts, ends, rows, keys = _inputs(q, k, key_scales, weights, starts, ends)
    if out is None:
        out = torch.empty((rows, int(topk)), dtype=torch.int32, device=q.device)
    out = _as(out, torch.int32, (rows, int(topk)), "out")
    rows_per_call = max(1, min(rows, int(logits_budget_bytes) // (keys * 4)))
    if logits_ws is None:
        logits_ws = torch.empty(rows_per_call * keys, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(HEADER_BYTES, dtype=torch.uint8, device=q.device)
    budget = min(int(logits_budget_bytes), logits_ws.numel() * logits_ws.element_size())
    _check(lib().mqa_topk_dense_baseline(_ptr(q), _ptr(k), _ptr(key_scales), _ptr(weights), _ptr(starts),
                                         _ptr(ends), _ptr(out), rows, keys, int(topk), _ptr(logits_ws), budget,
                                         _ptr(workspace), workspace.numel(), _stream(stream)),
           "mqa_topk_dense_baseline")
    return out


def alloc_host_staging(rows: int, keys: int, topk: int, device=None):
    """Device staging for mqa_topk_prefill_host (inputs, scales, output and
    workspace; caller owns it)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else int(device))
    n = ctypes.c_size_t()
    _check(lib().mqa_topk_host_staging_bytes(dev.index, int(rows), int(keys), int(topk), ctypes.byref(n)),
           "mqa_topk_host_staging_bytes")
    return torch.empty(n.value, dtype=torch.uint8, device=dev)


def mqa_topk_prefill_host(q, k, scales_ue8m0, weights, starts, ends, topk: int, staging, out, stream=None):
    """The fused op from host tensors (pinned for asynchronous copies): every
    copy, the scale decode and the kernel are enqueued by the C entry on
    `stream`; `out` (host int32 [rows, topk]) is valid once the stream has
    reached this point."""
    torch = _torch()
    rows, keys = int(q.shape[0]), int(k.shape[0])
    for t, name in ((q, "q"), (k, "k"), (scales_ue8m0, "scales_ue8m0"), (weights, "weights"), (starts, "starts"),
                    (ends, "ends"), (out, "out")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: a contiguous host tensor is expected")
    _check(lib().mqa_topk_prefill_host(_ptr(q), _ptr(k), _ptr(scales_ue8m0), _ptr(weights), _ptr(starts),
                                       _ptr(ends), _ptr(out), rows, keys, int(topk), _ptr(staging),
                                       staging.numel() * staging.element_size(), _stream(stream)),
           "mqa_topk_prefill_host")
    return out


def host_get_status(staging, rows: int, keys: int, topk: int, stream=None):
    """get_status for the workspace inside a mqa_topk_prefill_host staging buffer."""
    st = ctypes.c_int32(0)
    stats = (ctypes.c_int32 * len(STAT_NAMES))()
    _check(lib().mqa_topk_host_get_status(_ptr(staging), int(rows), int(keys), int(topk), ctypes.byref(st), stats,
                                          _stream(stream)), "mqa_topk_host_get_status")
    return int(st.value), dict(zip(STAT_NAMES, [int(v) for v in stats]))


def get_status(workspace, stream=None):
    """(status bits, {counter name: value}) of the last call on `workspace` (synchronises)."""
    st = ctypes.c_int32(0)
    stats = (ctypes.c_int32 * len(STAT_NAMES))()
    _check(lib().mqa_topk_get_status(_ptr(workspace), ctypes.byref(st), stats, _stream(stream)),
           "mqa_topk_get_status")
    return int(st.value), dict(zip(STAT_NAMES, [int(v) for v in stats]))
