"""Build libbsfp8.so in-tree with nvcc for sm_103a (no cmake, one translation
unit per .cu file, compiled in parallel, linked with the static CUDA runtime).

    python -m block_scaled_fp8_sm_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libbsfp8.so")
OBJ = os.path.join(HERE, "_build")
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["bsfp8_api.cu"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "bsfp8.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(OUT):
        return True
    t = os.path.getmtime(OUT)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return OUT
    os.makedirs(OBJ, exist_ok=True)
    nvcc = _nvcc()
    flags = GENCODE + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                       "-I", os.path.join(ROOT, "include")]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
        subprocess.run([nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj], check=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = OUT + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *GENCODE, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(OUT)
