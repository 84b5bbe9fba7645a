"""Build the in-tree CUDA libraries for sm_103a with nvcc (no cmake, one translation unit each):
libvt_attn.so, and libvt_attn_debug.so, the same source with VT_DEBUG (device index checks that report
VT_ERR_DEVICE_BOUNDS).  The two compile in parallel."""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libvt_attn.so")
LIB_DEBUG = os.path.join(PKG, "libvt_attn_debug.so")
SOURCES = [os.path.join(CSRC, "vt_attn_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("vt_attn_f32_2q.cuh", "vt_attn_bf16_2q.cuh", "vt_attn_common.cuh", "vt_attn_merge.cuh",
                                                  "vt_ptx.cuh")] + [
    os.path.join(os.path.dirname(PKG), "include", "vt_attn.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvt_attn.so")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in DEPS if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libvt_attn.so and libvt_attn_debug.so next to this file; returns the release library's path."""
    jobs = []
    for lib, extra in ((LIB, []), (LIB_DEBUG, ["-DVT_DEBUG"])):
        if force or not up_to_date(lib):
            tmp = lib + ".tmp"
            cmd = [nvcc(), *NVCC_FLAGS, *extra, "-o", tmp, *SOURCES]
            jobs.append((lib, tmp, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    for lib, tmp, proc in jobs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(lib)} ({proc.returncode}):\n{out}\n{err}")
        if verbose:
            print(err)
        os.replace(tmp, lib)
    return LIB
