"""Build libqp.so in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` compiles to an object in parallel, then nvcc links the
shared library next to this file.  Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libqp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]
if os.environ.get("QP_TRACE") == "1":   # compile the phase-trace hooks in (include/qp_debug.h)
    NVCC_FLAGS.append("-DQP_TRACE=1")


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libqp.so)")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                               + glob.glob(os.path.join(INCLUDE, "*.h")))


FLAGS_STAMP = os.path.join(BUILD_DIR, "flags.txt")


def up_to_date(flags=None) -> bool:
    """The library exists, is newer than every source and header, and was
    built with the same compiler flags."""
    if not os.path.exists(LIB_PATH):
        return False
    if flags is not None:
        if not os.path.exists(FLAGS_STAMP) or open(FLAGS_STAMP).read() != " ".join(flags):
            return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile every CUDA source and link libqp.so; returns its path."""
    flags = NVCC_FLAGS + list(extra_flags or [])
    if not force and up_to_date(flags):
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        jobs.append((src, obj, [nvcc] + ARCH + flags + ["-c", src, "-o", obj]))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(lambda j: _run(j[2]), jobs))
    if verbose:
        for (src, _, _), o in zip(jobs, outs):
            if o.strip():
                print(f"[{os.path.basename(src)}]\n{o}", file=sys.stderr)
    tmp = LIB_PATH + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-o", tmp] + [j[1] for j in jobs])
    os.replace(tmp, LIB_PATH)
    with open(FLAGS_STAMP, "w") as f:
        f.write(" ".join(flags))
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None))
