"""libnorm from a plain C program (tests/c_caller.c): the public header, device
memory from the CUDA runtime, no Python or PyTorch on the calling side.  On
the CPU the program is compiled as C99 with warnings as errors and linked
against libnorm.so, the oracle and the CUDA runtime; on a GPU it also runs,
and every output of a LayerNorm and a BatchNorm forward and backward must
match the CPU oracle within the fp32 parity bound."""
import os
import subprocess

import pytest

import oracle
from normalization_layernorm_rmsnorm_gb300 import build as nbuild

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_caller.c")


def _cuda_root():
    return os.path.dirname(os.path.dirname(os.path.realpath(nbuild.nvcc())))


def _compile(out_dir):
    lib = nbuild.build()
    olib = oracle.build()
    cuda = _cuda_root()
    cuda_lib = os.path.join(cuda, "lib64")
    dirs = [os.path.dirname(lib), os.path.dirname(olib), cuda_lib]
    exe = os.path.join(str(out_dir), "c_caller")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", SRC,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.dirname(oracle.__file__),
           "-I", os.path.join(cuda, "include"),
           "-L", dirs[0], "-lnorm", "-L", dirs[1], "-loracle", "-L", cuda_lib, "-lcudart", "-lm",
           "-Wl,-rpath," + ":".join(dirs), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_caller_matches_the_oracle(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    if r.returncode == 2:
        pytest.skip("needs a CUDA GPU")
    assert r.returncode == 0 and r.stdout.startswith("ok"), f"rc {r.returncode}\n{r.stdout}\n{r.stderr}"
