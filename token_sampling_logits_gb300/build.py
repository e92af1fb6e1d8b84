"""Builds libgsample.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

    python -m token_sampling_logits_gb300.build        # build if stale
    python -m token_sampling_logits_gb300.build -f     # force a rebuild
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgsample.so")
OBJ_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libgsample.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Compile the library (if stale, or forced). With out_dir, a variant with
    extra_flags (e.g. -DGSAMPLE_COUNT_BLOCKS) is built there instead, always,
    leaving the regular library alone; returns the path of the built .so."""
    lib_path = LIB if out_dir is None else os.path.join(out_dir, "libgsample.so")
    obj_dir = OBJ_DIR if out_dir is None else out_dir
    if out_dir is None and not force and not is_stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, res.stdout, res.stderr))
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    force = "-f" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else None
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra_flags=extra))
