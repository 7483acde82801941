"""Compile libmoe_layout.so (the C-ABI library) in-tree for sm_103a with nvcc.

The translation units are compiled in parallel and linked into
``combine_moe_layout_gb300/_lib/libmoe_layout.so``; a stamp of the sources,
headers and flags skips rebuilds that would change nothing.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libmoe_layout.so")
STAMP = os.path.join(LIBDIR, "libmoe_layout.stamp")

SOURCES = ["moe_layout.cu", "moe_dispatch.cu", "moe_layout_dispatch.cu", "moe_recv.cu", "moe_combine.cu",
           "moe_expert_stub.cu", "moe_route_stats.cu", "moe_expert.cu",
           "moe_expert_noalloc.cu", "moe_expert_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_layout.so")


def _inputs_hash(extra: list[str]) -> str:
    h = hashlib.sha256()
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))] + [os.path.join(INCLUDE, "moe_layout.h")]
    for path in files:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          lib_path: str | None = None) -> str:
    """Build the library (default: the in-tree _lib/libmoe_layout.so); extra_flags and
    lib_path build a variant elsewhere without touching the default one."""
    extra = list(extra_flags or [])
    lib = lib_path or LIB
    stamp = lib + ".stamp" if lib_path else STAMP
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    want = _inputs_hash(extra)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == want:
                return lib
    cc = nvcc()
    objdir = os.path.join(os.path.dirname(lib), "obj" if not lib_path else "obj_" + os.path.basename(lib))
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    res = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(want)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
