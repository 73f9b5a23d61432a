"""The C ABI from plain C: tests/c/roundtrip.c includes only uzip.h and the
CUDA runtime header and calls libuzip directly (cudaMalloc'd buffers, the
default stream). On the CPU the program must compile as C11 and link against
the built library (uzip.h is a C header, every function it uses is
exported); on a GPU it must round-trip its input bit-exactly."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "lossless_bf16_exponent_gb300")
CUDA = "/usr/local/cuda"


def _build(tmp_path, name="roundtrip"):
    from lossless_bf16_exponent_gb300 import build as B

    lib = B.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / name)
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", name + ".c"), "-o", exe,
           "-L", os.path.dirname(lib), "-luzip", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))
    assert os.path.exists(_build(tmp_path, "noalloc_reset"))


@pytest.mark.gpu
@pytest.mark.parametrize("n,chunk", [(1, 8), (1000003, 1024), (4 << 20, 256), (65537, 65536)])
def test_c_client_round_trip(tmp_path, uz, n, chunk):
    exe = _build(tmp_path)
    r = subprocess.run([exe, str(n), str(chunk)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "roundtrip ok" in r.stdout
