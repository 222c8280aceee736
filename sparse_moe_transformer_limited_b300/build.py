"""Compile the CUDA library (libbeam_moe.so) in-tree for sm_103a.

Run as `python -m sparse_moe_transformer_limited_b300.build` or call build().
nvcc cross-compiles without a GPU. The runtime is linked statically, so the
library loads on a machine without a driver (it only needs one to run).
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libbeam_moe.so")
SOURCES = ["beam_moe.cu"]
HEADERS = ["ptx.cuh", "kernels_gemm.cuh", "kernels_gemm_tm.cuh", "kernels_gemm_wide.cuh", "kernels_gemm_2sm.cuh",
           "kernels_combine.cuh", "kernels_ep.cuh",
           "kernels_permute.cuh", "kernels_quant.cuh", "kernels_router.cuh", "kernels_rows.cuh",
           "kernels_attn.cuh"]


def nvcc_cmd(out=LIB, extra=()):
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    return [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2", "-cudart", "static",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC,
            *extra, "-o", out] + [os.path.join(CSRC, s) for s in SOURCES]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "beam_moe.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    """Build libbeam_moe.so if a source is newer than it (or force)."""
    if not force and not _stale():
        return LIB
    cmd = nvcc_cmd(extra=["-Xptxas", "-v"] if verbose else [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
