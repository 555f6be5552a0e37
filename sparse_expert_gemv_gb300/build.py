"""Build libmoe_decode.so in-tree with nvcc for sm_103a (no cmake, one TU).

    python -m sparse_expert_gemv_gb300.build
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "moe_decode.cu")
OUT = os.path.join(HERE, "libmoe_decode.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def command(out: str = OUT, extra=()) -> list[str]:
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-cudart", "shared", f"-I{os.path.join(ROOT, 'include')}",
            f"-Xlinker", f"-rpath,{cuda_lib}", *extra, SRC, "-o", out]


def build(verbose: bool = False) -> str:
    tmp = OUT + ".tmp"
    cmd = command(tmp, ["-Xptxas", "-v"] if verbose else [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libmoe_decode.so")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
