"""Build ``libattn_b300.so`` in-tree with nvcc for sm_103a.

Usage: ``python -m io_aware_attention_03_b300.build [--force]``.  nvcc
cross-compiles without a GPU.  The library links the CUDA runtime as a shared
library (the same ``libcudart.so.13`` torch loads), so the library and torch
share one runtime and one context per device.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_PATH = os.path.join(HERE, "libattn_b300.so")
MAIN_SOURCE = os.path.join(CSRC, "attn_b300.cu")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  [os.path.join(ROOT, "include", "attn_b300.h")])


KERNEL_SOURCES = {
    "prefill": ("prefill.cuh", "ptx.cuh", "common.cuh"),
    "prefill_fp8": ("prefill.cuh", "ptx.cuh", "common.cuh"),
    "decode": ("decode.cuh", "ptx.cuh", "common.cuh"),
    "backward_dkdv": ("backward.cuh", "prefill.cuh", "ptx.cuh", "common.cuh"),
    "backward_dq": ("backward.cuh", "prefill.cuh", "ptx.cuh", "common.cuh"),
}


def _code_only(text: str) -> str:
    """Source text with C/C++ comments removed and whitespace collapsed."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def source_signature(kind: str) -> str:
    """Short hash of one kernel family's device code (comments and layout ignored).

    Ties a stored profiler figure (e.g. DRAM bytes per launch) to the code it
    measured: once the kernel's code changes, the figure no longer applies.
    """
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:12]


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in _sources())


def nvcc_command(output: str, extra=()) -> list:
    cuda_lib = "/usr/local/cuda/lib64"
    return [NVCC, *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "--shared", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-cudart", "shared",
            f"-Xlinker", f"-rpath,{cuda_lib}", "-I", os.path.join(ROOT, "include"),
            *extra, "-o", output, MAIN_SOURCE]


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else [])
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB_PATH)
