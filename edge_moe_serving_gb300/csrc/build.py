"""Build libmoe.so in-tree with nvcc for sm_103a (GB300).

    python edge_moe_serving_gb300/csrc/build.py [--force] [--ptxas-verbose]

A plain script (not imported through the package, whose import needs the
library that this script builds).
"""
import os
import subprocess
import sys

CSRC = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(CSRC)
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmoe.so")
SOURCES = ["moe_api.cu", "route_topk.cu", "route_tc.cu", "dispatch.cu", "bind.cu", "ffn.cu", "ffn_gemv.cu",
           "ffn_gemm.cu", "combine.cu", "ffn_noalloc.cu",
           "front_small.cu", "decode_layer.cu", "selftest.cu", "bandwidth.cu", "ffn_mxfp4.cu", "ffn_mxfp4_ring.cu", "ffn_fp4_gemm.cu", "prefill_stack.cu",
           "fp4_layer.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h", ".py"))]
    files.append(os.path.join(INCLUDE, "moe.h"))
    return files


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force=False, ptxas_verbose=False, quiet=True):
    """Compile every CUDA source into libmoe.so (one nvcc call, parallel TUs)."""
    if not force and up_to_date():
        return LIB
    home = cuda_home()
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [os.path.join(home, "bin", "nvcc"), "-shared", "-Xcompiler", "-fPIC,-O2", "-std=c++17", "-O3",
           "-lineinfo", ARCH, "--threads", "0", "-cudart", "shared", "-I", INCLUDE, "-I", CSRC,
           "-Xlinker", "-rpath," + os.path.join(home, "lib64")]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES] + ["-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building libmoe.so")
    if not quiet or ptxas_verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_verbose="--ptxas-verbose" in sys.argv, quiet=False)
    print(LIB)
