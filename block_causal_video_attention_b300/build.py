"""Build the CUDA library libod_attn.so in-tree (nvcc, sm_103a only).

    python -m block_causal_video_attention_b300.build
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libod_attn.so")
LIB_DEBUG = os.path.join(PKG, "libod_attn_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-Xptxas", "-v",
]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cuh", ".h")))


def needs_build() -> bool:
    return needs_build_of(LIB)


def needs_build_of(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    hdr = os.path.join(ROOT, "include", "od_attn.h")
    return any(os.path.getmtime(f) > t for f in sources() + [hdr])


def _nvcc(lib: str, extra, verbose: bool) -> str:
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [NVCC] + NVCC_FLAGS + list(extra) + ["-I", os.path.join(ROOT, "include"), "-o", tmp,
                                               os.path.join(CSRC, "od_api.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building %s" % os.path.basename(lib))
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """libod_attn.so, the library the binding loads."""
    if not force and not needs_build_of(LIB):
        return LIB
    return _nvcc(LIB, [], verbose)


def build_debug(force: bool = False, verbose: bool = False) -> str:
    """libod_attn_debug.so: the same sources with -DOD_DEBUG (device-side range checks)."""
    if not force and not needs_build_of(LIB_DEBUG):
        return LIB_DEBUG
    return _nvcc(LIB_DEBUG, ["-DOD_DEBUG"], verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
    if "--debug" in sys.argv:
        print(build_debug(force="--force" in sys.argv, verbose=True))
