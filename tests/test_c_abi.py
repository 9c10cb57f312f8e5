"""The C ABI used from a plain C program (tests/c/abi_smoke.c): include/kda.h compiles as
C11, the program links against libkda.so, and on a GPU it runs a prefill through the
device and the host-buffer entry points (bit-identical results) and checks status codes."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "kda_recurrent_state_gb300")
CUDA = "/usr/local/cuda"


def _compile(out_path):
    from kda_recurrent_state_gb300 import build

    build.build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cmd = [gcc, "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "abi_smoke.c"), "-L", PKG, "-lkda", "-L",
           os.path.join(CUDA, "lib64"), "-lcudart", "-lm", f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{CUDA}/lib64", "-o",
           out_path]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out_path


def test_header_is_c11_and_program_links(tmp_path):
    _compile(str(tmp_path / "abi_smoke"))


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    exe = _compile(str(tmp_path / "abi_smoke"))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "abi_smoke ok" in r.stdout, r.stdout + r.stderr
