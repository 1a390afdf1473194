"""Compile libattn_sink.so for sm_103a with nvcc (in-tree, no torch extension)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libattn_sink.so")
# Test build: the same sources with the bounded waits lowered to 2 ms and the
# hooks that let a test withhold one tile (exercises the timeout path).
TEST_LIB_PATH = os.path.join(LIB_DIR, "libattn_sink_test.so")
TEST_FLAGS = ["-DATTN_SINK_TEST_HOOKS", "-DATTN_SINK_WAIT_LIMIT_NS=2000000ull"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libattn_sink.so")


def _sources() -> list[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "attn_sink.h"))
    return files


def build(force: bool = False, verbose: bool = False, test: bool = False) -> str:
    """Build the shared library (or, with test=True, the test build) if any
    source is newer than it; return its path."""
    path = TEST_LIB_PATH if test else LIB_PATH
    srcs = _sources()
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= max(os.path.getmtime(s) for s in srcs)):
        return path
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = path + ".tmp"
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-shared", "-I", INCLUDE, *(TEST_FLAGS if test else []), "-o", tmp,
           os.path.join(CSRC, "attn_sink_api.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
