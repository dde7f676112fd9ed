"""The C ABI used from plain C: tests/c/abi_roundtrip.c is compiled as C99 by
gcc against include/moe_ep.h, libmoeep.so and the CUDA runtime's C API (no C++
and no Python on its path).  On any host the program must compile and link; on
a GPU it runs one HT forward (route with a node limit, receive-count query,
bf16 dispatch, combine) and checks the identity round trip, the routing
invariants and the row map itself."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_roundtrip.c")


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.isfile(os.path.join(c, "include", "cuda_runtime_api.h")):
            return c
    return None


def _compile(tmp_path):
    gcc = shutil.which("gcc")
    cuda = _cuda_home()
    if gcc is None or cuda is None:
        pytest.skip("gcc or the CUDA toolkit is missing")
    from combine_layout_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.isdir(d)), None)
    if cudalib is None:
        pytest.skip("no CUDA runtime library directory")
    exe = str(tmp_path / "abi_roundtrip")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           SRC, "-o", exe, "-L", libdir, "-lmoeep", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    _compile(tmp_path)


@pytest.mark.gpu
def test_c_program_round_trip(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
