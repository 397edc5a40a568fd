"""Builds libdflash.so (sm_103a) in the package directory.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
one shared library with the CUDA runtime linked statically.  Only the C ABI
declared in include/dflash.h is exported.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdflash.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, extra=(), out: str = LIB) -> str:
    """Builds the library at `out`; extra nvcc flags (e.g. -D...) build a
    variant in a build folder of its own."""
    build_dir = BUILD if out == LIB else out + ".build"
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    heads = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    heads.append(os.path.join(ROOT, "include", "dflash.h"))
    newest = max(os.path.getmtime(p) for p in srcs + heads + [__file__])
    if os.path.exists(out) and os.path.getmtime(out) > newest and not extra:
        return out
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra), build_dir), srcs))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print("built", out)
    return out


if __name__ == "__main__":
    args = sys.argv[1:]
    dest = LIB
    if len(args) >= 2 and args[0] == "--out":
        dest = os.path.abspath(args[1])
        args = args[2:]
    build(verbose=True, extra=args, out=dest)
