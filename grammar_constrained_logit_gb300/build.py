"""Build liblp.so, the CUDA library behind the C ABI in include/lp.h.

Compiles every ``csrc/*.cu`` for sm_103a only (one ``-gencode``), in parallel,
into ``_build/`` and links ``liblp.so`` next to this file.  No cmake, no torch
extension machinery: plain nvcc, so the same command works on the x86 build
container and on the Arm GPU host.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def _nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblp.so")
    return path


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (when stale) and return the path of liblp.so."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "lp.h")]
    objs, procs = [], []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"{src}:\n{out}")
        elif verbose and out:
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines: dict, sources=("sample.cu",), force: bool = False) -> str:
    """A test build: the given csrc sources compiled with extra preprocessor
    definitions and linked as ``_build/<name>/liblp.so``.  Test builds exercise
    paths that the product build cannot reach on demand (a bounded wait made to
    run out); the product library ``liblp.so`` is never one of them."""
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, name)
    os.makedirs(out_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, x) for x in sources]
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "lp.h")]
    lib = os.path.join(out_dir, "liblp.so")
    defs = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    stamp = os.path.join(out_dir, "defines.txt")
    same = os.path.exists(stamp) and open(stamp).read() == " ".join(defs)
    if force or not same or _stale(lib, srcs + headers):
        objs = []
        for src in srcs:
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
            subprocess.check_call([nvcc, *ARCH, *FLAGS, *defs, "-c", src, "-o", obj])
            objs.append(obj)
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
        with open(stamp, "w") as f:
            f.write(" ".join(defs))
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
