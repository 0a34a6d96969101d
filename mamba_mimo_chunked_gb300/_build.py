"""Build step of the CUDA library: one nvcc call, sm_103a only, in-tree."""

from __future__ import annotations

import os
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
SOURCES = [os.path.join(PKG_DIR, "csrc", "mmbf_kernels.cu")]
HEADERS = [os.path.join(REPO_DIR, "include", "mamba_mimo_bwd_fwd.h"),
           os.path.join(REPO_DIR, "include", "mamba_mimo_bwd_bwd.h"),
           os.path.join(PKG_DIR, "csrc", "mmbf_fast.cuh"),
           os.path.join(PKG_DIR, "csrc", "mmbf_tc.cuh"),
           os.path.join(PKG_DIR, "csrc", "mmbb.cuh")]
LIB_PATH = os.path.join(PKG_DIR, "libmmbf.so")
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    # The shared CUDA runtime: inside a process that already loaded one (e.g.
    # torch's), the library uses that same runtime instance, so streams and
    # events created there are valid handles here.
    "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB_PATH
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *NVCC_FLAGS, "-I", os.path.join(REPO_DIR, "include"), *SOURCES, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
