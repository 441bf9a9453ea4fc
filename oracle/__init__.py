"""CPU oracle (TEST INFRASTRUCTURE ONLY).

A plain fp64 C implementation of what the fused prefill selection computes
(see `mqa_oracle.c` for the definition and its sources).  It shares no code
with the CUDA library and imports nothing from it.  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may use it; the
product path never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mqa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmqa_oracle.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc into oracle/_build (portable flags only)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: str):
    """Open an oracle shared library and declare its entry points."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_ue8m0_decode.argtypes = [P, P, ctypes.c_int64]
    lib.oracle_head_dots.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, P]
    lib.oracle_run.argtypes = [P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
    lib.oracle_run.restype = ctypes.c_int
    lib.oracle_run_blocks.argtypes = [P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
    lib.oracle_run_blocks.restype = ctypes.c_int
    lib.oracle_run_masked.argtypes = [P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, P, ctypes.c_int64, P, P, ctypes.c_int]
    lib.oracle_run_masked.restype = ctypes.c_int
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_fold_prep.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]
    lib.oracle_fold_score.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_int64]
    lib.oracle_fold_score.restype = ctypes.c_double
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def e4m3_table(lib=None) -> np.ndarray:
    out = np.empty(256, np.float64)
    _load(lib).oracle_e4m3_table(_ptr(out))
    return out


def ue8m0_decode(groups: np.ndarray, lib=None) -> np.ndarray:
    g = _c(groups, np.uint8)
    assert g.ndim == 2 and g.shape[1] == 4
    out = np.empty(g.shape[0], np.float32)
    _load(lib).oracle_ue8m0_decode(_ptr(g), _ptr(out), g.shape[0])
    return out


def head_dots(q: np.ndarray, k: np.ndarray, row: int, key: int, lib=None) -> np.ndarray:
    q = _c(q, np.uint8)
    k = _c(k, np.uint8)
    heads, dim = q.shape[1], q.shape[2]
    out = np.empty(heads, np.float64)
    _load(lib).oracle_head_dots(_ptr(q), _ptr(k), heads, dim, row, key, _ptr(out))
    return out


FOLD_TERMS = 4


def e4m3_encode(x: float, lib=None) -> int:
    """e4m3fn code nearest to x (|x| <= 448), ties to even."""
    return int(_load(lib).oracle_e4m3_encode(ctypes.c_double(float(x))))


def fold_prep(q, w, terms=FOLD_TERMS, lib=None):
    """The folded query v = sum_h w_h q_h (fp32, fused multiply-add per head in
    head order) written as `terms` e4m3 vectors with power-of-two scales.
    Returns (codes [rows, terms, dim] uint8, exps [rows, terms] int32,
    v [rows, dim] float32, beta [rows] float64: 2-norm of the last residual)."""
    q = _c(q, np.uint8)
    w = _c(w, np.float32)
    rows, heads, dim = q.shape
    codes = np.empty((rows, terms, dim), np.uint8)
    exps = np.empty((rows, terms), np.int32)
    v = np.empty((rows, dim), np.float32)
    beta = np.empty(rows, np.float64)
    _load(lib).oracle_fold_prep(_ptr(q), _ptr(w), rows, heads, dim, terms, _ptr(codes), _ptr(exps), _ptr(v),
                                _ptr(beta))
    return codes, exps, v, beta


def fold_score(p, codes, exps, row, key, lib=None):
    """scale_j * (sum_t 2^e_t E(u_t) . E(k_j) + sum_h w_h |s_h|) / 2 in fp64."""
    q = _c(p.q, np.uint8)
    k = _c(p.k, np.uint8)
    g = _c(p.scales_ue8m0, np.uint8)
    w = _c(p.weights, np.float32)
    c = _c(codes, np.uint8)
    e = _c(exps, np.int32)
    return float(_load(lib).oracle_fold_score(_ptr(q), _ptr(k), _ptr(g), _ptr(w), _ptr(c), _ptr(e), q.shape[1],
                                              q.shape[2], c.shape[1], int(row), int(key)))


def run(p, rows=None, want_topk=True, want_scores=False, topk=None, nthreads=None, lib=None):
    """Run the oracle on problem `p` (a `synth.Problem`-like object) for the
    listed rows (default: all).  Returns (indices [n, topk] or None,
    scores [n, keys] fp64 or None)."""
    q = _c(p.q, np.uint8)
    k = _c(p.k, np.uint8)
    g = _c(p.scales_ue8m0, np.uint8)
    w = _c(p.weights, np.float32)
    s = _c(p.starts, np.int32)
    e = _c(p.ends, np.int32)
    rows = np.arange(q.shape[0], dtype=np.int64) if rows is None else _c(rows, np.int64)
    topk = int(p.topk if topk is None else topk)
    n = rows.shape[0]
    out = np.empty((n, topk), np.int32) if want_topk else None
    scores = np.empty((n, k.shape[0]), np.float64) if want_scores else None
    rc = _load(lib).oracle_run(_ptr(q), _ptr(k), _ptr(g), _ptr(w), _ptr(s), _ptr(e), _ptr(rows),
                            n, k.shape[0], q.shape[1], q.shape[2], topk,
                            _ptr(out) if out is not None else None,
                            _ptr(scores) if scores is not None else None,
                            int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_run failed with status {rc}")
    return out, scores


def run_blocks(p, btopk, rows=None, nthreads=None, lib=None):
    """Top `btopk` blocks of 8 keys per listed row by their largest score:
    [n, btopk] int32, block index relative to the row's first block
    (floor(start / 8)), best first (ties by block index), -1 padded."""
    q = _c(p.q, np.uint8)
    k = _c(p.k, np.uint8)
    g = _c(p.scales_ue8m0, np.uint8)
    w = _c(p.weights, np.float32)
    s = _c(p.starts, np.int32)
    e = _c(p.ends, np.int32)
    rows = np.arange(q.shape[0], dtype=np.int64) if rows is None else _c(rows, np.int64)
    n = rows.shape[0]
    out = np.empty((n, int(btopk)), np.int32)
    rc = _load(lib).oracle_run_blocks(_ptr(q), _ptr(k), _ptr(g), _ptr(w), _ptr(s), _ptr(e), _ptr(rows), n,
                                      k.shape[0], q.shape[1], q.shape[2], int(btopk), _ptr(out),
                                      int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_run_blocks failed with status {rc}")
    return out


def run_masked(p, mask, rows=None, want_topk=True, want_scores=False, topk=None, nthreads=None, lib=None):
    """Masked selection: mask [rows, words] uint32, bit (j / 8) % 32 of word
    j / 256 allows key j for the row.  Returns (indices, scores) as `run`."""
    q = _c(p.q, np.uint8)
    k = _c(p.k, np.uint8)
    g = _c(p.scales_ue8m0, np.uint8)
    w = _c(p.weights, np.float32)
    s = _c(p.starts, np.int32)
    e = _c(p.ends, np.int32)
    m = _c(mask, np.uint32)
    rows = np.arange(q.shape[0], dtype=np.int64) if rows is None else _c(rows, np.int64)
    topk = int(p.topk if topk is None else topk)
    n = rows.shape[0]
    out = np.empty((n, topk), np.int32) if want_topk else None
    scores = np.empty((n, k.shape[0]), np.float64) if want_scores else None
    rc = _load(lib).oracle_run_masked(_ptr(q), _ptr(k), _ptr(g), _ptr(w), _ptr(s), _ptr(e), _ptr(rows), n,
                                      k.shape[0], q.shape[1], q.shape[2], topk, _ptr(m), m.shape[1],
                                      _ptr(out) if out is not None else None,
                                      _ptr(scores) if scores is not None else None,
                                      int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_run_masked failed with status {rc}")
    return out, scores


def topk(p, rows=None, nthreads=None, lib=None):
    return run(p, rows, True, False, nthreads=nthreads, lib=lib)[0]


def logits(p, rows=None, nthreads=None, lib=None):
    return run(p, rows, False, True, nthreads=nthreads, lib=lib)[1]
