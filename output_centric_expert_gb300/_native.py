"""Compile and load the package's native libraries (in-tree, under ``_build/``).

Two shared libraries are built from ``csrc/``:

* ``libwarp_decode.so`` -- the C-ABI library: the two CUDA kernels
  (``moe_gate_up`` in wd_gate_up*.cu, ``moe_down`` in wd_down.cu), the C-ABI
  entry points and router (warp_decode.cu) and the host-side MXFP8 packer.
  Compiled by ``nvcc`` for sm_103a only, one translation unit per file, in
  parallel.
* ``libworkload.so`` -- the seeded synthetic input generator (plain C, gcc).

Nothing here falls back to another implementation: if a library is missing or
fails to load, the caller gets an exception.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD = os.path.join(PKG_DIR, "_build")
REPO = os.path.dirname(PKG_DIR)
INCLUDE = os.path.join(REPO, "include")

LIB_WARP_DECODE = os.path.join(BUILD, "libwarp_decode.so")
LIB_WORKLOAD = os.path.join(BUILD, "libworkload.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwarp_decode.so")
    return cand


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _cuda_sources() -> list[str]:
    names = ["warp_decode.cu", "wd_gate_up.cu", "wd_gate_up_fixed.cu", "wd_gate_up_grouped.cu",
             "wd_down.cu", "wd_down_grouped.cu", "pack.cpp"]
    return [os.path.join(CSRC, n) for n in names]


def _cuda_deps() -> list[str]:
    deps = _cuda_sources()
    for d in (CSRC, INCLUDE):
        deps += [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".h", ".cuh"))]
    return deps


def build_warp_decode(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile libwarp_decode.so (kernels + launchers + packer) for sm_103a."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and not _stale(LIB_WARP_DECODE, _cuda_deps()):
        return LIB_WARP_DECODE
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-Xcompiler", "-fPIC"]
    objs = []
    cmds = []
    for src in _cuda_sources():
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH_FLAGS, "-lineinfo", *common, "-c", src, "-o", obj]
            if verbose_ptxas:
                cmd.insert(1, "-Xptxas=-v")
        else:
            cmd = [nvcc, *common, "-x", "c++", "-c", src, "-o", obj]
        cmds.append(cmd)
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(_run, cmds))
    tmp = LIB_WARP_DECODE + ".tmp"
    _run([nvcc, *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB_WARP_DECODE)
    return LIB_WARP_DECODE


def build_workload(force: bool = False) -> str:
    """Compile libworkload.so (seeded input generator, plain C)."""
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(CSRC, "workload.c")
    if not force and not _stale(LIB_WORKLOAD, [src]):
        return LIB_WORKLOAD
    tmp = LIB_WORKLOAD + ".tmp"
    _run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", tmp, "-lm"])
    os.replace(tmp, LIB_WORKLOAD)
    return LIB_WORKLOAD


def load(path_builder) -> ctypes.CDLL:
    """Build if needed and load a library; raises if it cannot be loaded."""
    with _lock:
        key = path_builder.__name__
        if key not in _libs:
            path = path_builder()
            _libs[key] = ctypes.CDLL(path)
        return _libs[key]
