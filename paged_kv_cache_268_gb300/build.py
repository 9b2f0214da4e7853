"""Build libpkv.so (sm_103a) in-tree with nvcc.

The decode kernels are split over four translation units (element type x
kernel variant) plus the C-ABI front end, compiled in parallel and linked into
``paged_kv_cache_268_gb300/lib/libpkv.so``.  Run ``python -m
paged_kv_cache_268_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(OUT_DIR, "libpkv.so")
OBJ_DIR = os.path.join(ROOT, "_build", "pkv")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required to build libpkv)")


def _units():
    units = [("pkv_api", "pkv_api.cu", []), ("pkv_noalloc", "pkv_noalloc.cu", []),
             ("pkv_blocks", "pkv_blocks.cpp", []), ("pkv_decode_tc", "pkv_decode_tc.cu", [])]
    for bf in (0, 1):
        for mma in (0, 1):
            name = f"pkv_decode_{'bf16' if bf else 'f16'}_{'mma' if mma else 'simt'}"
            units.append((name, "pkv_decode_inst.cu",
                          [f"-DPKV_INST_BF16={bf}", f"-DPKV_INST_MMA={mma}"]))
    return units


def _sources():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pkv.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    cc = nvcc()
    common = [cc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(unit):
        name, src, defs = unit
        obj = os.path.join(OBJ_DIR, name + ".o")
        cmd = [*common, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    units = _units()
    with cf.ThreadPoolExecutor(max_workers=len(units)) as ex:
        results = list(ex.map(compile_one, units))
    if verbose or ptxas_info:
        for (name, _, _), (_, log) in zip(units, results):
            if log.strip():
                print(f"== {name}\n{log}", file=sys.stderr)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv))
