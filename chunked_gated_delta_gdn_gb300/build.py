"""Build libgdn.so in-tree with nvcc for sm_103a (GB300).

    python -m chunked_gated_delta_gdn_gb300.build [--force] [--verbose-ptxas] [--variant stamps]

Each ``csrc/*.cu`` file is compiled in parallel to an object file under
``chunked_gated_delta_gdn_gb300/_build/`` and linked into
``chunked_gated_delta_gdn_gb300/_build/libgdn.so`` (CUDA runtime linked
statically, so the library needs nothing but the driver at run time).

Diagnostic variants build the same sources with extra defines into
``_build/<variant>/libgdn.so``; nothing loads them but the tools that ask for them:
``stamps`` (-DGDN_CHUNK_STAMPS) records the chunk kernel's stage timestamps.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
VARIANTS = {"stamps": ["-DGDN_CHUNK_STAMPS"]}


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgdn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def lib_path(variant=None) -> str:
    return LIB if variant is None else os.path.join(BUILD, variant, "libgdn.so")


def up_to_date(variant=None) -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose_ptxas: bool, variant=None) -> str:
    out_dir = os.path.dirname(lib_path(variant))
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           *VARIANTS.get(variant, []), "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, res.stdout, res.stderr))
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, variant=None) -> str:
    """Compile (if stale) and return the path of libgdn.so (of a diagnostic variant)."""
    if variant is not None and variant not in VARIANTS:
        raise ValueError("unknown build variant %r" % variant)
    lib = lib_path(variant)
    if not force and up_to_date(variant):
        return lib
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, variant), srcs))
    tmp = lib + ".%d.tmp" % os.getpid()
    cmd = [nvcc_path(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (res.stdout, res.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--variant", choices=sorted(VARIANTS))
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, variant=args.variant))
