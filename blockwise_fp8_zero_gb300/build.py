"""Build libfp8z.so (sm_103a CUDA kernels + host C ABI) in-tree.

nvcc compiles the .cu files for exactly one target, sm_103a; g++ compiles the
host-only C++; nvcc links the shared library with a static CUDA runtime.  The
translation units compile in parallel; nothing is rebuilt when sources, headers
and flags are unchanged.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8z.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["step.cu", "aux.cu", "fold.cu", "rowwise.cu"]
CPP_SOURCES = ["host.cpp", "plan.cpp"]
HEADERS = [os.path.join(CSRC, "fp8z_device.cuh"), os.path.join(CSRC, "fp8z_host.h"),
           os.path.join(INCLUDE, "fp8z.h")]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(_cuda_home(), "bin", "nvcc")


def _commands():
    cuda = _cuda_home()
    inc = ["-I", INCLUDE, "-I", CSRC]
    cmds = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "--fmad=false",
               "-Xcompiler", "-fPIC,-ffp-contract=off,-fvisibility=hidden", "-Xptxas", "-v", *inc,
               "-c", os.path.join(CSRC, src), "-o", obj]
        cmds.append((src, obj, cmd))
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math",
               "-fvisibility=hidden",
               "-Wall", "-Wextra", *inc, "-I", os.path.join(cuda, "include"),
               "-c", os.path.join(CSRC, src), "-o", obj]
        cmds.append((src, obj, cmd))
    return cmds


def _stamp(cmds) -> str:
    h = hashlib.sha256()
    for _, _, cmd in cmds:
        h.update(" ".join(cmd).encode())
    for path in [os.path.join(CSRC, s) for s in CU_SOURCES + CPP_SOURCES] + HEADERS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    cmds = _commands()
    stamp = _stamp(cmds)
    stamp_file = os.path.join(BUILD_DIR, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    procs = [(src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
             for src, _, cmd in cmds]
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(f"--- {src}\n{out}")
        if p.returncode != 0:
            failed.append(src)
        elif src.endswith(".cu"):
            with open(os.path.join(BUILD_DIR, src + ".ptxas.txt"), "w") as f:
                f.write(out)
    if failed:
        raise RuntimeError(f"fp8z build failed: {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [_nvcc(), *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in cmds]]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
