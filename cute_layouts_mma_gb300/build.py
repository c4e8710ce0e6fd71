"""Build the CUDA library in-tree: csrc/*.cu -> _build/libtn_gemm.so (sm_103a only).

Each translation unit is compiled in parallel with nvcc, then linked with the
static CUDA runtime.  Re-running is cheap: nothing is rebuilt when no source
or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtn_gemm.so")
# Test-only variants.  timeout_inject: one pipeline arrival is withheld so that a
# bounded wait runs out (exercises the abandon path).  scale_copy: the block-scaled
# instances move their scales with tcgen05.cp instead of tcgen05.st (the pages' copy
# instruction, kept as a tested compile-time alternative).
VARIANTS = {"timeout_inject": ["-DTN_TIMEOUT_INJECT"], "scale_copy": ["-DTN_SCALE_COPY"]}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def lib_path(variant: str = "") -> str:
    if not variant:
        return LIB
    return os.path.join(BUILD, variant, f"libtn_gemm_{variant}.so")


def up_to_date(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Build the library (variant "" is the product; others are test builds)."""
    lib = lib_path(variant)
    if not force and up_to_date(variant):
        return lib
    outdir = os.path.dirname(lib)
    os.makedirs(outdir, exist_ok=True)
    nvcc = _nvcc()
    extra = VARIANTS[variant] if variant else []

    def compile_one(src):
        obj = os.path.join(outdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(_sources())) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for obj, log in results:
            sys.stderr.write(f"--- {os.path.basename(obj)}\n{log}")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
