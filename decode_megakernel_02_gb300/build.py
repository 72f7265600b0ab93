"""Compile libmk.so in-tree for sm_103a (nvcc for the CUDA units, g++ for the
host-only units), in parallel, without CMake."""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libmk.so")
BUILD = os.path.join(ROOT, "_build")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CU_SRCS = ["mk_vm_bf16.cu", "mk_vm_fp16.cu", "mk_vm_int8.cu", "mk_vm_int4.cu", "mk_vm_fp8.cu", "mk_vm_common.cu",
           "mk_runtime.cu",
           "mk_static.cu", "mk_prefill.cu"]
CPP_SRCS = ["mk_host.cpp", "mk_schedule.cpp", "mk_validate.cpp"]


def _sources():
    return [os.path.join(CSRC, f) for f in CU_SRCS + CPP_SRCS] + [
        os.path.join(CSRC, f) for f in ("mk_internal.h", "mk_host.h", "mk_vm.cuh", "mk_prefill.h")] + [os.path.join(INCLUDE, "mk.h")]


def up_to_date():
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force=False, verbose=False):
    """Build decode_megakernel_02_gb300/libmk.so; returns its path."""
    if not force and up_to_date():
        return OUT
    os.makedirs(BUILD, exist_ok=True)
    inc = ["-I" + INCLUDE, "-I" + CSRC]
    procs = []
    objs = []
    for f in CU_SRCS:
        o = os.path.join(BUILD, f + ".o")
        cmd = [NVCC, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", *inc, "-c",
               os.path.join(CSRC, f), "-o", o]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(o)
    cxx = shutil.which("g++") or "g++"
    for f in CPP_SRCS:
        o = os.path.join(BUILD, f + ".o")
        cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-Wall", *inc, "-I" + os.path.join(CUDA_HOME, "include"),
               "-c", os.path.join(CSRC, f), "-o", o]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(o)
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(" ".join(cmd) + "\n" + text)
        elif verbose and text.strip():
            sys.stderr.write(text)
    if failed:
        raise RuntimeError("libmk build failed:\n" + "\n".join(failed))
    tmp = OUT + ".tmp"
    link = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("libmk link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
