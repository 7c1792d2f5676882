"""In-tree build of libmla_decode.so for sm_103a.

CUDA sources go through nvcc (one -gencode: arch=compute_103a, code=sm_103a),
host C++ through g++, all translation units in parallel, then one shared
link with the static CUDA runtime. Run as ``python -m
mla_decode_attention_09_gb300.build`` or call ``build()``.
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmla_decode.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

CUDA_SOURCES = ["stage1.cu", "stage1_umma.cu", "stage1_umma_a16.cu", "stage1_umma_pairs.cu", "reduce.cu", "noalloc.cu"]
CXX_SOURCES = ["plan.cpp", "capi.cpp"]
GENCODE = "arch=compute_103a,code=sm_103a"


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "mla_decode.h")]
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _sources()) and os.path.getmtime(__file__) <= t


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library if any source changed; returns the .so path."""
    if not force and up_to_date():
        return LIB_PATH
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = shutil.which("nvcc") or nvcc
    os.makedirs(BUILD_DIR, exist_ok=True)
    common_inc = ["-I", INCLUDE, "-I", CSRC]
    jobs = []
    objs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [nvcc, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "--expt-relaxed-constexpr", *common_inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, src))
        objs.append(obj)
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = ["g++", "-O2", "-fPIC", "-std=c++17", "-Wall", *common_inc, "-I", os.path.join(cuda, "include"),
               "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, src))
        objs.append(obj)
    procs = [(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True), src, cmd)
             for cmd, src in jobs]
    failed = []
    for p, src, cmd in procs:
        out, _ = p.communicate()
        if verbose or ptxas_info or p.returncode != 0:
            if out:
                sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"compilation failed for {failed}")
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, "-gencode", GENCODE, "-shared", "-o", tmp, *objs, "-lpthread"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB_PATH)
