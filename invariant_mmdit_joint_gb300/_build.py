"""Builds librlk_joint_attn.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel with the same
strict-math flags (no --use_fast_math; IEEE division and square root; no
flush-to-zero), then linked into one shared library next to this file.
"""

from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB_NAME = "librlk_joint_attn.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
STRICT = ["-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-fmad=true"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return path


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def source_hash() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def build(out_dir: str | None = None, extra_flags: list[str] | None = None,
          lib_name: str = LIB_NAME, srcs: list[str] | None = None, verbose: bool = False) -> str:
    """Compile and link; returns the path of the shared library."""
    out_dir = out_dir or PKG
    obj_dir = os.path.join(out_dir, "_build")
    os.makedirs(obj_dir, exist_ok=True)
    extra = list(extra_flags or [])
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE] + STRICT + extra
    tag = " ".join(["sm_103a"] + STRICT + extra)
    defs = [f'-DRLK_SOURCE_HASH="{source_hash()}"', f'-DRLK_BUILD_FLAGS="{tag}"']
    srcs = srcs or sources()

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc()] + flags + defs + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    lib = os.path.join(out_dir, lib_name)
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
