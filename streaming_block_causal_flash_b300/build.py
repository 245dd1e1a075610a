"""Build the native library in-tree: ``libws_b300.so`` next to this file.

nvcc compiles every ``csrc/*.cu`` for sm_103a only and links them into one
shared object with the CUDA runtime linked statically; the C ABI is
``include/ws.h``.  ``build(debug=True)`` builds ``libws_b300_debug.so`` from
the same sources with ``-DWS_DEBUG=1``: every index a kernel computes for a
global-memory access is bounds-checked, and a failed check is recorded in the
device error word and the access skipped (never a trap).  The binding loads
the debug library when the environment variable ``WS_DEBUG=1`` is set.
Run as ``python -m streaming_block_causal_flash_b300.build [--debug]``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
LIB_NAME = "libws_b300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libws_b300_debug.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(PKG_DIR, "csrc", "*.cu")))


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = sources() + glob.glob(os.path.join(PKG_DIR, "csrc", "*.h")) + \
        glob.glob(os.path.join(PKG_DIR, "csrc", "*.cuh")) + [os.path.join(ROOT, "include", "ws.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and not _stale(path):
        return path
    cmd = [nvcc_path(), "-O3", "-std=c++17", *ARCH_FLAGS, "-lineinfo",
           "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared",
           "-I", os.path.join(ROOT, "include"),
           *(["-DWS_DEBUG=1"] if debug else []),
           "-o", path + ".tmp", *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(path + ".tmp", path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
