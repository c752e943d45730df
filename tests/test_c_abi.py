"""The C ABI from plain C: tests/c_abi/tide_c_client.c is compiled with gcc
against include/tide.h and linked to libtide.so (no Python or C++ between).
On the CPU it builds host-only plans and checks geometry, errors and the
schedule planners; on a GPU it also runs the fold and the placements and
compares them bit for bit with the CPU oracle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "tide_c_client.c")


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.isdir(os.path.join(cand, "include")):
            return cand
    pytest.skip("CUDA toolkit not found")


def _compile(tmp_path, gpu: bool) -> str:
    from all_gather_gb300 import build
    build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(build.LIB)
    exe = str(tmp_path / ("client_gpu" if gpu else "client"))
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), SRC,
           "-o", exe, "-L", libdir, "-ltide"]
    rpath = [libdir]
    if gpu:
        import oracle
        oracle.load()
        cuda = _cuda_home()
        cudalib = os.path.join(cuda, "lib64")
        cmd[1:1] = ["-DTIDE_C_CLIENT_GPU", "-I", os.path.join(cuda, "include")]
        cmd += ["-L", os.path.dirname(oracle.LIB_PATH), "-ltide_oracle", "-L", cudalib, "-lcudart"]
        rpath += [os.path.dirname(oracle.LIB_PATH), cudalib]
    cmd.append("-Wl,-rpath," + ":".join(rpath))
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_client_host(tmp_path):
    exe = _compile(tmp_path, gpu=False)
    res = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0 and res.stdout.strip() == "OK", res.stderr


@pytest.mark.gpu
def test_c_client_gpu(tmp_path):
    exe = _compile(tmp_path, gpu=True)
    res = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == "OK", res.stderr
