"""Compile the CUDA sources into the in-tree shared library (sm_103a only)."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libncp_attn.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    # Share the process's CUDA runtime (the one torch loads) so the current
    # device and stream handles mean the same thing on both sides.
    "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.h"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, quiet: bool = False, extra_flags=None) -> str:
    """Build ``_lib/libncp_attn.so`` with nvcc if it is missing or stale."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(extra_flags or []), "-I", INCLUDE, "-o", tmp, *sources()]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if not quiet and res.stderr.strip():
        print(res.stderr.strip())
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def build_variant(name: str, extra_flags) -> str:
    """Build the same sources with extra compile flags into
    ``_lib/libncp_attn_<name>.so`` (test builds that exercise rare paths);
    rebuilt when missing or stale."""
    path = os.path.join(LIB_DIR, f"libncp_attn_{name}.so")
    if os.path.exists(path) and all(os.path.getmtime(f) <= os.path.getmtime(path)
                                    for f in _inputs()):
        return path
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-o", tmp, *sources()]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    os.replace(tmp, path)
    return path
