"""Build libkvq.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into quantized_kv_cache_quantize_gb300/libkvq.so
(static CUDA runtime; the driver is reached through the runtime's entry-point
query, so no -lcuda).  No fast-math: the quantizer relies on IEEE fp32
division, rounding and ties-to-even.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvq.so")
SOURCES = ["kvq_api.cu", "kvq_quant.cu", "kvq_quant_mma.cu", "kvq_attn.cu", "kvq_attn_exact.cu", "kvq_attn_kch.cu",
           "kvq_attn_pair.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


CHECKED_LIB = os.path.join(PKG, "libkvq_checked.so")


def _compile(src: str, verbose_ptxas: bool, checked: bool = False) -> str:
    out_dir = os.path.join(BUILD, "checked") if checked else BUILD
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    if checked:
        cmd[1:1] = ["-DKVQ_DEBUG_BOUNDS"]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, checked: bool = False) -> str:
    """libkvq.so, or with checked=True libkvq_checked.so: the same sources with
    -DKVQ_DEBUG_BOUNDS, whose kernels test their global-memory indices (a
    debugging build; see kvq_debug_bounds_site in include/kvq.h)."""
    os.makedirs(os.path.join(BUILD, "checked") if checked else BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, checked), SOURCES))
    lib = CHECKED_LIB if checked else LIB
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))
