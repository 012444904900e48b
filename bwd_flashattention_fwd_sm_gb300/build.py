"""Builds libgbattn.so in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library under ``bwd_flashattention_fwd_sm_gb300/_build/``.  The same sources
are also built with GBATTN_CHECKED=1 into libgbattn_checked.so, whose kernels
compare every device-computed index with its tensor's extent before the access
(selected at load time by the environment variable GBATTN_CHECKED=1).  A stamp
of the sources' contents and the flags decides whether a rebuild is needed.

Run ``python -m bwd_flashattention_fwd_sm_gb300.build [--force] [--ptxas-v]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgbattn.so")
LIB_CHECKED = os.path.join(BUILD, "libgbattn_checked.so")

SOURCES = ["api.cu", "sched.cu", "bwd_aux.cu", "simt_attn.cu", "tma_host.cu", "tc_fwd.cu", "tc_bwd.cu", "tc_dq.cu",
           "noalloc.cu", "ln.cu", "fp8.cu", "tc_bwd256.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgbattn.so")


def _sources():
    return [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]


def _stamp(extra) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    for name in sorted(os.listdir(INCLUDE)):
        if name.endswith(".h"):
            h.update(name.encode())
            with open(os.path.join(INCLUDE, name), "rb") as f:
                h.update(f.read())
    h.update(" ".join(ARCH + FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    """Compile and link both libraries if their sources changed; return the
    path of the plain one (LIB_CHECKED is the checked one)."""
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    stamp = _stamp(extra)
    stamp_file = os.path.join(BUILD, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(LIB_CHECKED) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB
    variants = (("obj", [], LIB), ("obj_checked", ["-DGBATTN_CHECKED=1"], LIB_CHECKED))
    for sub, _, _ in variants:
        os.makedirs(os.path.join(BUILD, sub), exist_ok=True)
    cc = nvcc()

    def compile_one(job):
        sub, defs, src = job
        obj = os.path.join(BUILD, sub, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return sub, src, obj, r

    jobs = [(sub, defs, src) for sub, defs, _ in variants for src in _sources()]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, jobs))
    for sub, src, obj, r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({sub}):\n{r.stdout}\n{r.stderr}")
        if (not quiet or ptxas_verbose) and sub == "obj":
            sys.stderr.write(r.stderr)
    for sub, _, lib in variants:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *[obj for s, _, obj, _ in results if s == sub]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_verbose="--ptxas-v" in sys.argv, quiet=False)
    print(LIB)
