"""Build libswa.so in-tree: nvcc for sm_103a, translation units compiled in parallel.

`build(checked=True)` builds libswa_checked.so from the same sources with
SWA_CHECKS=1: its kernels test every global load and store against the
extent of its tensor and report an access outside it as SWA_ERR_BOUNDS
instead of making it (include/swa.h, swa_workspace_status).  It is a
testing build; nothing loads it unless asked to (swa.checked_lib())."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libswa.so")
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libswa_checked.so")
SOURCES = ["swa_api.cpp", "swa_fwd.cu", "swa_fwd_pair.cu", "swa_bwd_dkv.cu", "swa_bwd_dq.cu", "swa_aux.cu",
           "swa_noalloc.cu", "swa_host.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libswa")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "swa.h")]
    return [f for f in files if os.path.isfile(f)]


def is_stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile every translation unit for sm_103a and link libswa.so (or,
    with `checked`, the bounds-checked libswa_checked.so); returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if not force and not is_stale(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    defines = ["-DSWA_CHECKS=1"] if checked else []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
