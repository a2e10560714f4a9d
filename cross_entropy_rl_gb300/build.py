"""Build the in-tree shared library ``_lib/libll_gb300.so`` for sm_103a.

Every CUDA translation unit under ``csrc/`` is compiled in parallel with
nvcc (one ``-gencode``: compute_103a -> sm_103a) and linked into one shared
library with the C ABI declared in ``include/ll_linear_logp.h``.

    python -m cross_entropy_rl_gb300.build [-v] [--ptxas-verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libll_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

SOURCES = ["capi.cu", "logits_kernels.cu", "gemm_tc.cu", "gemm_tf32.cu",
           "aux_kernels.cu", "noalloc.cu"]
HEADERS = ["ll_device.cuh", "ll_internal.h", "epilogue.cuh", "gemm_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(ROOT, "include", "ll_linear_logp.h"), __file__]
    if not _stale(obj, deps) and not ptxas_verbose:
        return obj, ""
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    objs = [o for o, _ in results]
    if verbose or ptxas_verbose:
        for (o, log), s in zip(results, SOURCES):
            if log:
                print(f"--- {s}\n{log}")
    if _stale(LIB_PATH, objs):
        # every symbol must resolve at link time (a missing definition is a
        # build error, not a load-time error)
        cmd = [nvcc(), *ARCH, "-shared", "-Xlinker", "--no-undefined", "-o", LIB_PATH, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return LIB_PATH


if __name__ == "__main__":
    p = build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas-verbose" in sys.argv)
    print(p)
