"""Compile the CUDA library in-tree: libb300attn.so next to this file, sm_103a only.

    python -m exact_transformer_attention_flashattention_b300.build [--force] [--debug]

`--debug` builds libb300attn_debug.so instead: the same library compiled with
-DB300ATTN_DEBUG, whose kernels also check caller data they otherwise clamp
(kv_len, cu_seqlens) and their own index invariants, and report a failed check
through attn_device_status (see csrc/debug.cuh).  The binding loads it when
the environment variable B300ATTN_DEBUG is 1.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libb300attn.so")
LIB_DEBUG = os.path.join(HERE, "libb300attn_debug.so")
SOURCE = os.path.join(CSRC, "b300attn.cu")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libb300attn.so")


def _inputs():
    files = [os.path.join(INCLUDE, "b300attn.h")]
    files += [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
              if f.endswith((".cu", ".cuh", ".h"))]
    return files


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def nvcc_command(out: str, debug: bool = False) -> list:
    """The nvcc command line that builds the library (or its debug variant) into `out`."""
    return [_nvcc(), *FLAGS, *(["-DB300ATTN_DEBUG"] if debug else []), *ARCH, "-o", out, SOURCE]


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build the shared library (or its debug variant) if any source is newer;
    return its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(debug):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, debug)
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose:
        sys.stdout.write(res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
