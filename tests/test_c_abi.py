"""The C ABI from a plain C11 program (tests/c_abi/decode_c.c): built with gcc
against include/pkv.h, libpkv.so, the CUDA runtime and the oracle's C source,
with no C++, PyTorch or binding in between.

On the CPU the program is compiled and linked with warnings as errors (the
header is valid C and every symbol it uses resolves); on the GPU it runs the
append, decode, set-workspace, no-alloc and fused-step calls on one ragged
batch and compares them with the oracle (see the program's header)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from paged_kv_cache_268_gb300 import _binding as B
from paged_kv_cache_268_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "decode_c.c")
ORACLE_SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nv = shutil.which("nvcc")
    if nv:
        return os.path.dirname(os.path.dirname(os.path.realpath(nv)))
    pytest.skip("no CUDA toolkit headers")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    build.build()
    lib = B.library_path()
    cuda = cuda_home()
    exe = str(tmp_path_factory.mktemp("c_abi") / "decode_c")
    cudalib = os.path.join(cuda, "lib64")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           SRC, ORACLE_SRC, "-o", exe,
           lib, f"-Wl,-rpath,{os.path.dirname(lib)}",
           "-L", cudalib, "-lcudart", f"-Wl,-rpath,{cudalib}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(program):
    assert os.access(program, os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,kernel,split,group,variant", [
    (0, 0, 0, 1, 0),      # fp16 MHA: CUDA cores, the library's partition
    (1, 0, 0, 4, 1),      # bf16 GQA 4: mma.sync
    (0, 0, 256, 4, 1),    # forced 256-token partitions: up to 11 per sequence
    (1, 0, 0, 32, 1),     # the widest group
    (1, 3, 0, 4, 2),      # the tcgen05 kernel
    (0, 3, 512, 16, 2),
])
def test_c_program_matches_the_oracle(program, dtype, kernel, split, group, variant):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([program, str(dtype), str(kernel), str(split), str(group)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = r.stdout.strip().splitlines()[-1]
    assert line.startswith("OK "), line
    fields = dict(kv.split("=") for kv in line.split()[1:])
    assert int(fields["variant"]) == variant
    if split:
        assert int(fields["splits"]) == -(-2600 // split)
