"""Build libkvc.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into one shared
library next to this file. Run `python -m kv_cache_compression_snapkv_gb300._build`.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvc.so")
LIB_CHECKED = os.path.join(PKG, "libkvc_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]
SOURCES = ["api.cu", "score.cu", "score_tc.cu", "acumul_tc.cu", "topk.cu", "quant.cu", "decode.cu",
           "noalloc.cu"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, extra, obj_dir: str = OBJ) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    if os.path.exists(obj):
        os.remove(obj)   # never link an object left from an earlier build
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 or not os.path.exists(obj):
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, extra=(), checked: bool = False) -> str:
    """Compile every CUDA source and link libkvc.so (libkvc_checked.so with
    checked=True: device-side index checks, KVC_CHECKED=1); returns the library path."""
    obj_dir = OBJ + ("_checked" if checked else "")
    lib = LIB_CHECKED if checked else LIB
    flags = list(extra) + (["-DKVC_CHECKED=1"] if checked else [])
    os.makedirs(obj_dir, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, obj_dir), SOURCES))
    cmd = [nvcc(), *ARCH, "-shared", "-o", lib + ".tmp", *objs, "-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(lib + ".tmp", lib)
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    if any(a in ("-h", "--help") for a in sys.argv[1:]):
        print("usage: python -m kv_cache_compression_snapkv_gb300._build [--checked] "
              "[extra nvcc flags ...]\n  --checked  build libkvc_checked.so (KVC_CHECKED=1: "
              "device-side checks of caller-given indices)")
        sys.exit(0)
    args = [a for a in sys.argv[1:] if a != "--checked"]
    build(verbose=True, extra=args, checked="--checked" in sys.argv[1:])
