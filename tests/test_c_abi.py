"""The C ABI from C: tests/c_abi_client.c is compiled with gcc as C99 against
include/tb.h alone and linked with libtb.so.

Without a GPU it runs the argument checks, which return before any CUDA call.
On the GPU it also runs a softmax backward and a LayerNorm backward through the C
entry points and compares them with the CPU oracle (linked into the client).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_client.c")


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()
    import ln_backward_gb300
    return ln_backward_gb300


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _compile(tmp_path, with_cuda):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / ("c_abi_client_gpu" if with_cuda else "c_abi_client"))
    pkg = os.path.join(ROOT, "ln_backward_gb300")
    cmd = [gcc, "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-Wno-unused-parameter",
           f"-I{os.path.join(ROOT, 'include')}", SRC, "-o", exe,
           f"-L{pkg}", "-ltb", f"-Wl,-rpath,{pkg}", "-lm"]
    if with_cuda:
        cuda = _cuda_home()
        orc = os.path.join(ROOT, "oracle")
        cmd[1:1] = ["-DWITH_CUDA", f"-I{os.path.join(cuda, 'include')}"]
        cmd += [f"-L{orc}", "-loracle", f"-Wl,-rpath,{orc}",
                f"-L{os.path.join(cuda, 'lib64')}", "-lcudart",
                f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stdout + p.stderr
    return exe


def test_c_client_argument_checks(built, tmp_path):
    exe = _compile(tmp_path, with_cuda=False)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "argument checks through the C ABI: ok" in p.stdout


@pytest.mark.gpu
def test_c_client_runs_kernels_against_the_oracle(built, tmp_path):
    exe = _compile(tmp_path, with_cuda=True)
    p = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "softmax bwd" in p.stdout and "LayerNorm bwd" in p.stdout
