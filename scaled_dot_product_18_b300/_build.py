"""Compile the CUDA library libattn.so in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libattn.so")
SOURCES = [os.path.join(CSRC, f) for f in ("attn_fwd_sm103.cu", "attn_bwd_sm103.cu", "attn_decode_sm103.cu",
                                           "gemm_sm103.cu", "attn_api.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("ptx_sm103.cuh", "attn_internal.h")] + [os.path.join(INCLUDE, "attn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


# The wait-timeout test library: the same sources compiled with
# SDP18_WAIT_TEST (5 ms wait limit, a producer stall hook and two test-only
# exports).  Only tests load it; the product library never contains the hook.
WAIT_TEST_LIB = os.path.join(PKG, "libattn_waittest.so")


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def _compile(lib: str, defines: list[str], verbose: bool) -> str:
    tmp = lib + ".tmp.%d" % os.getpid()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", *defines,
           "-I" + INCLUDE, "-o", tmp, *SOURCES, "-Xlinker", "-rpath=" + cuda_lib]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build(LIB):
        return LIB
    return _compile(LIB, [], verbose)


def build_wait_test(force: bool = False) -> str:
    if not force and not needs_build(WAIT_TEST_LIB):
        return WAIT_TEST_LIB
    return _compile(WAIT_TEST_LIB, ["-DSDP18_WAIT_TEST"], False)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
