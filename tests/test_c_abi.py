"""The C ABI from C: tests/c_abi/vt_attn_c_smoke.c is compiled with gcc as C99 against
include/vt_attn.h and linked with libvt_attn.so, then run."""

from __future__ import annotations

import os
import shutil
import subprocess

import pytest

import scaled_dot_product_vt_gb300 as vt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "vt_attn_c_smoke.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(out: str, with_cuda: bool) -> None:
    vt.build()
    libdir = os.path.dirname(vt.LIB)
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), SRC,
           "-o", out, "-L", libdir, "-lvt_attn", f"-Wl,-rpath,{libdir}"]
    if with_cuda:
        cmd[1:1] = ["-DVT_WITH_CUDA", "-I", os.path.join(CUDA, "include")]
        cmd += ["-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True)


def _run(exe: str) -> subprocess.CompletedProcess:
    return subprocess.run([exe], capture_output=True, text=True, timeout=120)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_c_consumer_host_checks(tmp_path):
    exe = str(tmp_path / "vt_attn_c_smoke")
    _build(exe, with_cuda=False)
    r = _run(exe)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_c_consumer_on_gpu(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "vt_attn_c_smoke_gpu")
    _build(exe, with_cuda=True)
    r = _run(exe)
    assert r.returncode == 0, r.stderr
