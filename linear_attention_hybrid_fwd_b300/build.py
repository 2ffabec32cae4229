"""Build step for liblightning_attn.so (nvcc, sm_103a only).

``python -m linear_attention_hybrid_fwd_b300.build`` compiles every ``csrc/*.cu``
into ``liblightning_attn.so`` inside the package directory, so the built library
travels with the source tree.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "liblightning_attn.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *FLAGS, *sources(), "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


TIMELINE_LIB = os.path.join(PKG, "liblightning_attn_timeline.so")


def build_timeline(force: bool = False) -> str:
    """The same sources with -DLA_TIMELINE: the prefill kernel stamps its pipeline
    events (see timeline.py).  A separate library; the product library is unchanged."""
    if not force and os.path.exists(TIMELINE_LIB) and os.path.exists(LIB) and \
            os.path.getmtime(TIMELINE_LIB) >= os.path.getmtime(build()):
        return TIMELINE_LIB
    tmp = TIMELINE_LIB + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, *ARCH, *FLAGS, "-DLA_TIMELINE", *sources(), "-o", tmp])
    os.replace(tmp, TIMELINE_LIB)
    return TIMELINE_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
