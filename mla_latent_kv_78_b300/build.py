"""Build libmla_b300.so in-tree with nvcc for sm_103a.

Usage: python -m mla_latent_kv_78_b300.build [--debug]
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmla_b300.so")
SOURCES = ["mla_api.cu", "append.cu", "absorb.cu", "absorb_tc.cu", "decode_simt.cu", "decode_tc.cu",
           "decode_noalloc.cu", "gemm_tc.cu", "prefill_tc.cu", "stage_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for p in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if p and os.path.exists(p):
            return p
    return "nvcc"


def is_current(lib: str, newest_source: float, flags: str) -> bool:
    """The library is current only if it is newer than every source and was built with the
    same extra flags (a stamp beside it, lib + ".flags", records them)."""
    stamp = lib + ".flags"
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        built_with = f.read()
    return os.path.getmtime(lib) >= newest_source and built_with == flags


def build(verbose: bool = False, extra=None) -> str:
    """Compile every .cu under csrc/ into one shared library. Returns its path."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    newest = max(os.path.getmtime(p) for p in srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC)])
    hdr = os.path.join(os.path.dirname(HERE), "include", "mla.h")
    newest = max(newest, os.path.getmtime(hdr), os.path.getmtime(__file__))
    flags = " ".join(extra or [])
    stamp = LIB + ".flags"
    if is_current(LIB, newest, flags):
        return LIB
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-Xptxas", "-v" if verbose else "-O3",
           "-o", LIB + ".tmp", *srcs, *(extra or [])]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libmla_b300.so")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(LIB + ".tmp", LIB)
    with open(stamp, "w") as f:
        f.write(flags)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
