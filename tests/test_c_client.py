"""A plain C program drives the library through include/kvsel.h alone (tests/c_client.c).

On the CPU: the header compiles as C and the program links against libkvsel.so and the CUDA
runtime.  On a GPU: the program runs score -> top-k -> compact and checks what the method fixes
(unit row mass, the planted key first, the top-k property, bit-exact gathered rows from device and
from pinned host memory, pageable memory refused before any launch).
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client.c")


def _cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _build(out_dir):
    from attention_kv_cache_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    lib_dir = os.path.dirname(build.LIB)
    cuda_lib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                 os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                                 os.path.join(cuda, "targets", "x86_64-linux", "lib")) if os.path.isdir(d)), None)
    if cuda_lib is None:
        pytest.skip("no CUDA runtime library directory")
    exe = os.path.join(out_dir, "c_client")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", lib_dir, "-lkvsel", "-L", cuda_lib, "-lcudart", "-lm",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_build(str(tmp_path)))


@pytest.mark.gpu
def test_c_client_runs(tmp_path, cuda):
    exe = _build(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "c client ok" in r.stdout
