"""Build the CUDA library in-tree: nvcc for sm_103a only, translation units
compiled in parallel, then linked into `_build/libmqatopk.so` with the CUDA
runtime linked statically (the driver entry points are resolved at run time).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmqatopk.so")
# (source, object, extra flags): the fused kernel is compiled for 32-head key
# selection with the direct head sum (8-row blocks), for 32-head key selection
# with the relu fold on the tensor core (6-row blocks), for 64 index heads per
# query row, and once each for block selection (top blocks of 8 keys), masked
# selection, and the 8-row key selection whose parked epilogue warps select
# rows in pairs (few-block calls; it also holds the logits instantiation and
# the allocation-free scratch).  The block and masked
# compilations form every relu on the FMA pipe: for them that measured faster
# (1.2% and 3.2% at 1M keys) than the default quarter on the ALU pipe.
SOURCES = [("mqa_fused.cu", "mqa_fused.o", []), ("mqa_fused.cu", "mqa_fused_fold.o", ["-DMQA_FOLD=1"]),
           ("mqa_fused.cu", "mqa_fused_h64.o", ["-DMQA_HEADS=64"]),
           ("mqa_fused.cu", "mqa_fused_blocks.o", ["-DMQA_BLOCKS=1", "-DMQA_RELU_ALU_CHUNKS=0"]),
           ("mqa_fused.cu", "mqa_fused_masked.o", ["-DMQA_MASKED=1", "-DMQA_RELU_ALU_CHUNKS=0"]),
           ("mqa_fused.cu", "mqa_fused_pairs.o", ["-DMQA_PAIR_HELPERS=1"]),
           ("mqa_gather.cu", "mqa_gather.o", []), ("mqa_aux.cu", "mqa_aux.o", []),
           ("mqatopk_api.cu", "mqatopk_api.o", [])]
HEADERS = ["mqa_internal.h", "ptx.cuh", "mqa_fold.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(extra=()):
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    # the compile flags live in this file: a change to it rebuilds every object
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "mqatopk.h"),
                                                       os.path.abspath(__file__)]
    objs, jobs = [], []
    for src, obj, defs in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, obj)
        objs.append(o)
        if force or _stale(o, [s, *hdrs]):
            jobs.append([nvcc(), *_flags(extra_flags), *defs, "-c", s, "-o", o])
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            res = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for c, r in zip(jobs, res):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(c) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {c[-3]}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
