"""Build libec.so in-tree: the CUDA kernels for sm_103a (nvcc) and the host codec (g++).

    python -m lossless_entropy_coded_gb300.build
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libec.so")
BUILD = os.path.join(HERE, "_build")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc") if os.path.exists(os.path.join(CUDA_HOME, "bin", "nvcc")) else "nvcc"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))] + [os.path.join(HERE, "..", "include", "ec.h")]


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return OUT
    os.makedirs(BUILD, exist_ok=True)
    inc = ["-I", os.path.join(HERE, "..", "include"), "-I", CSRC]
    k_obj = os.path.join(BUILD, "ec_kernels.o")
    h_obj = os.path.join(BUILD, "ec_host.o")
    jobs = [
        [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", *inc, "-c",
         os.path.join(CSRC, "ec_kernels.cu"), "-o", k_obj],
        ["g++", "-O3", "-std=c++17", "-fPIC", "-pthread", "-Wall", f"-I{CUDA_HOME}/include", *inc, "-c",
         os.path.join(CSRC, "ec_host.cpp"), "-o", h_obj],
    ]
    procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for j in jobs]
    for j, p in zip(jobs, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(j)}\n{out}")
        if verbose and out:
            print(out)
    tmp = OUT + f".tmp{os.getpid()}"
    link = [NVCC, *ARCH, "-shared", "-o", tmp, k_obj, h_obj, "-Xcompiler", "-pthread"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    os.replace(tmp, OUT)
    return OUT


def clean() -> None:
    shutil.rmtree(BUILD, ignore_errors=True)
    if os.path.exists(OUT):
        os.remove(OUT)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
