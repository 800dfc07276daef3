"""The C ABI from a plain C program (tests/c_client/tsx_client.c), built
with gcc against include/tsx.h and libtsx.so: the header is valid C and the
boundary works without Python.  On the CPU the client runs its host-side
checks (status codes, planning without a GPU); on a GPU also an fp32 fma
compared bit for bit with the C library's fmaf."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    import __graft_entry__

    __graft_entry__.build()
    import pipelined_elementwise_streaming_gb300 as tsx

    libdir = os.path.dirname(tsx.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_client") / "tsx_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", os.path.join(ROOT, "tests", "c_client", "tsx_client.c"),
           f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(CUDA, 'include')}", "-o", exe,
           f"-L{libdir}", "-l:libtsx.so", f"-Wl,-rpath,{libdir}",
           f"-L{os.path.join(CUDA, 'lib64')}", "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_host_checks(client):
    r = subprocess.run([client, "--no-gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout


@pytest.mark.gpu
def test_c_client_on_the_gpu(client):
    from tests import _gpu

    _gpu.need_gpu()
    r = subprocess.run([client], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok   fma equals fmaf bit for bit" in r.stdout
