"""Builds the in-tree shared library libds_verify.so for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked with
`nvcc -shared`.  The output lives next to this file (lib/), so the library
the tests and benchmark load is the one built from this tree.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "lib")
LIB_NAME = "libds_verify.so"
SOURCES = ["abi.cpp", "verify_attn.cu", "verify_tc.cu", "topk_gather.cu",
           "accept.cu", "accept_static.cu", "kv_commit.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", "-I" + INCLUDE, "-I" + CSRC]


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    srcs = [os.path.join(CSRC, s) for s in SOURCES
            if os.path.exists(os.path.join(CSRC, s))]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
            if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "ds.h"))
    return srcs, deps


def up_to_date() -> bool:
    p = lib_path()
    if not os.path.exists(p):
        return False
    t = os.path.getmtime(p)
    srcs, deps = _inputs()
    return all(os.path.getmtime(f) <= t for f in srcs + deps +
               [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return lib_path()
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, "_obj")
    os.makedirs(obj_dir, exist_ok=True)
    srcs, _ = _inputs()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-x", "cu", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path() + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path())
    return lib_path()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
