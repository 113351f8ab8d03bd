"""Compile libsarbp.so in-tree with nvcc for sm_103a (GB300).

The two translation units compile in parallel; the CUDA runtime is linked
statically so the library needs only the NVIDIA driver at run time.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsarbp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
_lock = threading.Lock()


def nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    default = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(default):
        return default
    raise RuntimeError("nvcc not found: libsarbp needs the CUDA toolkit to build")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + [os.path.join(INCLUDE, "sarbp.h"), os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    with _lock:
        if not force and not is_stale():
            return LIB
        os.makedirs(BUILD_DIR, exist_ok=True)
        cc = nvcc()
        procs = []
        objs = []
        for src in sources():
            obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [cc] + FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        failed = []
        for cmd, p in procs:
            out, _ = p.communicate()
            if verbose or p.returncode != 0:
                print(out.decode(errors="replace"))
            if p.returncode != 0:
                failed.append(" ".join(cmd))
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp = LIB + f".tmp{os.getpid()}"
        link = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        subprocess.run(link, check=True)
        os.replace(tmp, LIB)
        return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
