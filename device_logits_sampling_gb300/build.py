"""Build the sampling library in-tree for sm_103a (GB300).

Produces device_logits_sampling_gb300/_lib/libarcsample.so from csrc/: one
nvcc process per translation unit, all at once (the six kernel sets
dominate the build), then one link.  Runs on any host with nvcc (no GPU
needed).
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
SOURCES = [os.path.join(CSRC, f) for f in ("kernels_bf16.cu", "kernels_bf16_hist.cu", "kernels_f32.cu",
                                            "kernels_f32_hist.cu", "kernels_f16.cu", "kernels_f16_hist.cu",
                                            "arc_sample.cu", "arc_decode.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libarcsample.so")


def build(verbose: bool = False, extra: list[str] | None = None, out: str | None = None) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    target = out or LIB
    objdir = target + ".obj"
    os.makedirs(objdir, exist_ok=True)
    nvcc = nvcc_path()
    common = [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
              "-Xptxas", "-v" if verbose else "-O3", *(extra or [])]
    jobs = []
    for src in SOURCES:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *common, "-c", "-o", obj, src]
        jobs.append((cmd, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    failed = None
    for cmd, _, proc in jobs:
        so, se = proc.communicate()
        if proc.returncode != 0 and failed is None:
            failed = (proc.returncode, cmd, so + se)
        elif verbose:
            sys.stderr.write(se)
    if failed is not None:
        sys.stderr.write(failed[2])
        raise RuntimeError(f"nvcc failed ({failed[0]}): {' '.join(failed[1])}")
    link = [nvcc, *ARCH, "-shared", "-o", target + ".tmp", *[obj for _, obj, _ in jobs]]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc link failed ({res.returncode}): {' '.join(link)}")
    os.replace(target + ".tmp", target)
    shutil.rmtree(objdir, ignore_errors=True)
    return target


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
