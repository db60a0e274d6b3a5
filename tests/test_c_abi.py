"""The C ABI used from C: include/moe.h compiles as strict C99 and a C program links
against libmoe.so (CPU); the program runs a small layer through raw device buffers and
checks its own results (GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "layer_from_c.c")
PKG = os.path.join(ROOT, "combine_moe_route_softmax_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cuda_lib_dir():
    for d in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib", "lib"):
        if os.path.exists(os.path.join(CUDA, d, "libcudart.so")):
            return os.path.join(CUDA, d)
    pytest.skip("no libcudart.so under CUDA_HOME")


def _build(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = os.path.join(PKG, "libmoe.so")
    if not os.path.exists(lib):
        from combine_moe_route_softmax_gb300 import build
        build.build()
    exe = str(tmp_path / "layer_from_c")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", PKG, "-lmoe", "-L", _cuda_lib_dir(), "-lcudart",
           "-Wl,-rpath," + PKG]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_is_c99_and_links(tmp_path):
    _build(tmp_path)


@pytest.mark.gpu
def test_layer_from_c(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _build(tmp_path)
    env = dict(os.environ, LD_LIBRARY_PATH=PKG + ":" + _cuda_lib_dir() + ":" + os.environ.get("LD_LIBRARY_PATH", ""))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
