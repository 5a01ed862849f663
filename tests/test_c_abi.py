"""The C ABI from plain C: tests/c_abi/worked_example.c (C11, the CUDA runtime
for device memory, no Python or PyTorch on the path) compiles and links
against include/pkv.h and libpkv.so on any machine, and on a GPU runs the
pages' worked example end to end."""
import os
import shutil
import subprocess

import pytest

from paged_kv_prep_gb300 import build as pbuild

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_abi", "worked_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    pbuild.build()
    lib_dir = os.path.dirname(pbuild.LIBRARY)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "worked_example")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", "-I", pbuild.INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe,
           "-L", lib_dir, "-lpkv", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    exe = _compile(str(tmp_path))
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_program_runs_worked_example(tmp_path):
    exe = _compile(str(tmp_path))
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip() == "ok"
