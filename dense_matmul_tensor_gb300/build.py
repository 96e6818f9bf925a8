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
SOURCES = [os.path.join(CSRC, "bmm_api.cu"), os.path.join(CSRC, "attn_api.cu"),
           os.path.join(CSRC, "host_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("bmm_kernel.cuh", "ptx.cuh", "attn_kernel.cuh")] + [
    os.path.join(ROOT, "include", "bmm.h")]
OBJDIR = os.path.join(LIBDIR, "obj")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-DNDEBUG", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return exe


COMPILE = ["-O3", "-DNDEBUG", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden"]


def compile_commands(extra=()) -> list:
    """One nvcc command per translation unit (run in parallel)."""
    return [[nvcc(), *ARCH, *COMPILE, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o",
             os.path.join(OBJDIR, os.path.basename(src) + ".o")] for src in SOURCES]


def link_command(out: str = LIB) -> list:
    return [nvcc(), *ARCH, "-shared", "-o", out,
            *[os.path.join(OBJDIR, os.path.basename(s) + ".o") for s in SOURCES]]


def command(out: str = LIB, extra=()) -> list:
    """Single-command form (compile and link every source in one nvcc call)."""
    return [nvcc(), *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-o", out,
            *SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library unless it is newer than every source; return its path."""
    return finish(start(force=force, verbose=verbose))


class _Build:
    def __init__(self, procs, tmp):
        self.procs, self.tmp = procs, tmp


def start(force: bool = False, verbose: bool = False):
    """Start compiling every translation unit in parallel; None if current."""
    os.makedirs(OBJDIR, exist_ok=True)
    if not force and up_to_date():
        return None
    procs = []
    for cmd in compile_commands():
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append(subprocess.Popen(cmd))
    return _Build(procs, LIB + f".tmp{os.getpid()}")


def finish(job) -> str:
    if job is not None:
        for p in job.procs:
            if p.wait() != 0:
                raise subprocess.CalledProcessError(p.returncode, "nvcc")
        subprocess.run(link_command(job.tmp), check=True)
        os.replace(job.tmp, LIB)
    return LIB
