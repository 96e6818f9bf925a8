"""Build the in-tree GPU library ``_lib/libdmt_bmm.so`` for sm_103a with nvcc.

The shared library exports the C ABI of ``include/bmm.h``.  It links the CUDA
runtime statically and reaches the driver's tensor-map encoder through the
runtime's driver-entry-point query, so loading it needs no GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libdmt_bmm.so")
SOURCES = [os.path.join(CSRC, "bmm_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("bmm_kernel.cuh", "ptx.cuh")] + [
    os.path.join(ROOT, "include", "bmm.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-DNDEBUG", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return exe


def command(out: str = LIB, extra=()) -> list:
    return [nvcc(), *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-o", out,
            *SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library unless it is newer than every source; return its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = command(tmp)
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def start(force: bool = False):
    """Start the build in the background; returns a Popen or None if current."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and up_to_date():
        return None
    return subprocess.Popen(command(LIB + f".tmp{os.getpid()}"))


def finish(proc) -> str:
    if proc is not None:
        rc = proc.wait()
        if rc != 0:
            raise subprocess.CalledProcessError(rc, "nvcc")
        os.replace(LIB + f".tmp{os.getpid()}", LIB)
    return LIB
