"""Build ``libfp8lin.so`` in-tree with nvcc for sm_103a (no torch extension).

Each CUDA translation unit compiles in parallel; the shared library links the
CUDA runtime statically, so loading it needs no GPU driver (calls then fail
with FP8_ERR_CUDA).  Usage: ``python -m fp8_mixed_precision_history_gb300.build``.
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8lin.so")
SOURCES = ["fp8lin_api.cu", "cast_kernels.cu", "gemm_tcgen05.cu", "noalloc_cast.cu", "mx_kernels.cu",
           "grad_allreduce.cu"]
HEADERS = [os.path.join(CSRC, "state.cuh"), os.path.join(CSRC, "tc_ptx.cuh"), os.path.join(INCLUDE, "fp8lin.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
                     "-Wall", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _obj(src):
    return os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return all(os.path.getmtime(d) <= t for d in deps)


def start_compiles(verbose=False):
    """Start one nvcc per translation unit; returns [(src, Popen)]."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    for s in SOURCES:
        cmd = [nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + \
              ["-c", os.path.join(CSRC, s), "-o", _obj(s)]
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    return procs


def finish(procs):
    errors = []
    logs = []
    for s, p in procs:
        out, _ = p.communicate()
        logs.append(out.decode(errors="replace"))
        if p.returncode != 0:
            errors.append(f"--- {s} ---\n" + out.decode(errors="replace"))
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [_obj(s) for s in SOURCES]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return "\n".join(logs)


def build(verbose=False):
    log = finish(start_compiles(verbose))
    if verbose:
        print(log)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
