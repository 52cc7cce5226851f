"""The C ABI from C: tests/c/c_abi_prefill.c calls include/ple.h directly
(no Python in the loop) and checks every result against the oracle, which
it links as test infrastructure.  Without a GPU the program is only
compiled and linked, which checks that the header is plain C and that the
library exports what it declares; on a GPU it runs."""

import os
import shutil
import subprocess

import pytest
import torch

from layer_gram_embedding_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_program(tmp_path):
    lib = build.build()
    exe = str(tmp_path / "c_abi_prefill")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror",
           os.path.join(ROOT, "tests", "c", "c_abi_prefill.c"),
           os.path.join(ROOT, "oracle", "ple_oracle.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", os.path.dirname(lib), "-lple", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(CUDA, "lib64"),
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_compiles_and_links(tmp_path):
    compile_program(tmp_path)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_c_program_matches_the_oracle(tmp_path):
    exe = compile_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
