"""Builds the CUDA library libssm_scan.so in-tree (sm_103a only).

    python -m selective_state_space_111_b300.build

nvcc compiles csrc/ssm_scan_api.cu (forward), csrc/ssm_bwd_api.cu (backward)
and csrc/ssm_prologue_api.cu (prologue), which include their kernel headers,
into one shared library with the CUDA runtime linked statically, so the .so loads on a
machine without a GPU as well (for symbol checks) and needs nothing from the
environment at run time beyond the NVIDIA driver.

build_debug() compiles the same sources with SSM_DEBUG_BOUNDS defined into
libssm_scan_debug.so: the forward kernels check every global access and
bulk copy against its tensor's extent (a test-only build, loaded by the
tests that exercise it).

build_alu() compiles csrc/alu_rates.cu, the benchmark's throughput
microbenchmark of the update's instruction kinds, into its own small
libssm_alu.so (never loaded by the library or the tests).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libssm_scan.so")
SOURCES = [os.path.join(HERE, "csrc", f) for f in ("ssm_scan_api.cu", "ssm_bwd_api.cu",
                                                   "ssm_prologue_api.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in
                  ("bidir_kernel.cuh", "bwd_kernel.cuh", "prologue_kernel.cuh",
                   "scan_ops.cuh", "internal.h", "tc_ops.cuh")] + [
                  os.path.join(ROOT, "include", "ssm_scan.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
ALU_LIB = os.path.join(HERE, "libssm_alu.so")
DEBUG_LIB = os.path.join(HERE, "libssm_scan_debug.so")
ALU_SRC = os.path.join(HERE, "csrc", "alu_rates.cu")


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build(lib=LIB):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force=False, verbose=False, extra=(), lib=LIB):
    if not force and not needs_build(lib):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES, *extra]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


def build_debug(force=False):
    return build(force=force, extra=("-DSSM_DEBUG_BOUNDS",), lib=DEBUG_LIB)


def build_alu(force=False):
    if not force and os.path.exists(ALU_LIB) and os.path.getmtime(ALU_LIB) >= os.path.getmtime(ALU_SRC):
        return ALU_LIB
    tmp = ALU_LIB + ".tmp%d" % os.getpid()
    subprocess.check_call([nvcc(), *ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static", "-o", tmp,
                           ALU_SRC])
    os.replace(tmp, ALU_LIB)
    return ALU_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    build_alu(force="--force" in sys.argv)
    build_debug(force="--force" in sys.argv)
    print(LIB)
