"""Build the CUDA library in place: nvcc for sm_103a, one object per translation
unit compiled in parallel, linked into precision_gemm_gb300/libprecision_gemm.so
with the CUDA runtime linked statically (the library then loads on machines
without a GPU driver, and only the C-ABI symbols are exported)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libprecision_gemm.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["sgemm_api.cu", "ffma_kernel.cu", "tc_kernel.cu", "tc2_kernel.cu", "aux_kernels.cu"]
# Host-only C++ (the CPU co-worker of the hybrid column split), compiled by the host compiler.
HOST_SOURCES = ["host_sgemm.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]
# gnu++17 with explicit FMA contraction; no -march: the same flags build on x86 and Arm.
HOST_FLAGS = ["-O3", "-std=gnu++17", "-fPIC", "-fopenmp", "-ffp-contract=fast", "-fvisibility=hidden"]


def _cxx() -> str:
    return os.environ.get("CXX", "g++")


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "precision_gemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    for src in HOST_SOURCES:
        obj = os.path.join(BUILD, src.replace(".cpp", ".o"))
        objs.append(obj)
        cmd = [_cxx(), *HOST_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = LIB + ".tmp%d" % os.getpid()
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-lgomp",
            "-Xlinker", "-Bsymbolic", "-Xlinker", "--exclude-libs,ALL"]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    return LIB


PROBES = ("fma_ceiling", "tf32_ceiling")


def build_probe(name: str = "fma_ceiling", force: bool = False) -> str:
    """Compile a throughput probe (a small executable): the register-only FMA
    ceiling or the shared-memory-resident tcgen05 TF32 ceiling."""
    src = os.path.join(HERE, "probes", name + ".cu")
    binary = os.path.join(HERE, "probes", name)
    deps = [src] + ([os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "internal.h")] if name == "tf32_ceiling" else [])
    if not force and os.path.exists(binary) and all(os.path.getmtime(binary) >= os.path.getmtime(d) for d in deps):
        return binary
    subprocess.run([_nvcc(), *ARCH, "-O3", "-std=c++17", "-o", binary, src], check=True)
    return binary


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
