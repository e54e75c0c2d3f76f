"""Builds libsbp.so in-tree with nvcc for sm_103a (one object per .cu, compiled in parallel).

Variants of the same sources (each its own objects and library, selected at import time
by the SBP_LIBRARY_VARIANT environment variable):
  ""         libsbp.so          the library
  "checked"  libsbp_checked.so  guard zones after every workspace region, verified after
                                each call (SBP_ERR_WORKSPACE_OVERRUN); -DSBP_CHECKED
  "nvtx"     libsbp_nvtx.so     NVTX ranges per call and phase; -DSBP_NVTX
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsbp.so")
SOURCES = ["sbp_api.cu", "sbp_simt.cu", "sbp_tc.cu", "sbp_mlp.cu", "sbp_attn.cu", "sbp_attn_fused.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include"),
         "--expt-relaxed-constexpr"]
VARIANTS = {"": [], "checked": ["-DSBP_CHECKED"], "nvtx": ["-DSBP_NVTX"]}


def current_variant() -> str:
    """The variant this process loads (SBP_LIBRARY_VARIANT, default "")."""
    return os.environ.get("SBP_LIBRARY_VARIANT", "")


def lib_path(variant: str = "") -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown library variant {variant!r} (one of {sorted(VARIANTS)})")
    return LIB if not variant else os.path.join(PKG, f"libsbp_{variant}.so")


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsbp.so")
    return exe


def _compile(src: str, extra, obj_dir: str) -> str:
    out = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "sbp.h"),
                                                                 os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build_library(force: bool = False, extra=(), variant: str | None = None) -> str:
    """Compile every CUDA source of the library and link libsbp.so, or the variant's
    library (by default the one this process loads); returns its path."""
    if variant is None:
        variant = current_variant()
    lib = lib_path(variant)
    if not force and not _stale(lib):
        return lib
    obj_dir = os.path.join(OBJ, variant) if variant else OBJ
    os.makedirs(obj_dir, exist_ok=True)
    flags = VARIANTS[variant] + list(extra)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, obj_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(force=True))
