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
# the same library with the one-launch kernel's per-CTA timeline compiled in
# (-DMOE_TIMELINE: globaltimer stamps per CTA and phase, written to a
# caller-supplied buffer by moe_decode_layer_timeline); never loaded by the
# package itself
OUT_TIMELINE = os.path.join(HERE, "libmoe_decode_timeline.so")
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


def build(verbose: bool = False, timeline: bool = False) -> str:
    out = OUT_TIMELINE if timeline else OUT
    tmp = out + ".tmp"
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DMOE_TIMELINE"] if timeline else [])
    cmd = command(tmp, extra)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(out)}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, out)
    return out


def stale(path: str) -> bool:
    """True when `path` is missing or older than a CUDA source or header."""
    if not os.path.exists(path):
        return True
    srcs = [os.path.join(HERE, "csrc", f) for f in os.listdir(os.path.join(HERE, "csrc"))]
    srcs += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    return os.path.getmtime(path) < max(os.path.getmtime(f) for f in srcs)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, timeline="--timeline" in sys.argv))
