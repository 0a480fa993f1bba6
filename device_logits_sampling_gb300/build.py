"""Build the sampling library in-tree for sm_103a (GB300).

Produces device_logits_sampling_gb300/_lib/libarcsample.so from csrc/ with
one nvcc invocation.  Runs on any host with nvcc (no GPU needed).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libarcsample.so")
SOURCES = [os.path.join(CSRC, "arc_sample.cu"), os.path.join(CSRC, "arc_decode.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libarcsample.so")


def build(verbose: bool = False, extra: list[str] | None = None, out: str | None = None) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    target = out or LIB
    cmd = [
        nvcc_path(), *ARCH, "-O3", "-std=c++17", "-lineinfo",
        "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC,
        "-Xptxas", "-v" if verbose else "-O3",
        *(extra or []),
        "-o", target + ".tmp", *SOURCES,
    ]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed ({res.returncode}): {' '.join(cmd)}")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(target + ".tmp", target)
    return target


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
