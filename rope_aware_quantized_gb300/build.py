"""Builds the CUDA library libbgtq.so in-tree for sm_103a (GB300).

Three translation units are compiled in parallel with nvcc and linked into
one shared library exporting the C ABI declared in include/bgtq.h.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libbgtq.so")
# the BGTQ_DEBUG_BOUNDS build: every record and table index range-checked
# (a failure sets BGTQ_STATUS_BOUNDS and skips the access)
LIB_DEBUG = os.path.join(BUILD, "debug_bounds", "libbgtq_debug_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

SOURCES = [
    ("bgtq_host.cpp", []),
    ("codec.cu", ["--fmad=false"]),
    ("codec_bulk_k1.cu", ["--fmad=false"]),
    ("codec_bulk_k2.cu", ["--fmad=false"]),
    ("codec_bulk_k3.cu", ["--fmad=false"]),
    ("decode_attn.cu", []),
    ("decode_attn_paged.cu", []),
    ("decode_attn_noalloc.cu", []),
    ("fidelity.cu", []),
    ("prefill_attn.cu", []),
    ("prefill_chunk.cu", []),
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbgtq")
    return exe


def _compile(src: str, extra: list, verbose_ptxas: bool, outdir: str = BUILD) -> str:
    obj = os.path.join(outdir, src + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-std=c++17", "-O3", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC] + ARCH + extra
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def sources_newer_than(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "bgtq.h"), __file__]
    return any(os.path.getmtime(f) > t for f in files)


def build(force: bool = False, verbose_ptxas: bool = False, debug_bounds: bool = False) -> str:
    """Compile (if needed) and return the path of libbgtq.so (or, with
    debug_bounds, of the range-checked BGTQ_DEBUG_BOUNDS build)."""
    lib = LIB_DEBUG if debug_bounds else LIB
    if not force and not sources_newer_than(lib):
        return lib
    outdir = os.path.dirname(lib)
    os.makedirs(outdir, exist_ok=True)
    defs = ["-DBGTQ_DEBUG_BOUNDS"] if debug_bounds else []
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s[0], s[1] + defs, verbose_ptxas, outdir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
