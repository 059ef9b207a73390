"""Build libpagedkv.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel to an object file under
``_build/`` (the host-only block manager, ``kvmgr.cpp``, with the host C++
compiler); the objects link into ``paged_kv_decode_14_gb300/libpagedkv.so``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "api_noalloc.cu", "append.cu", "attn_simt.cu", "attn_tc.cu", "prefill.cu", "rope_append.cu", "kvmgr.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")


def cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("no host C++ compiler found (g++)")


def _flags(verbose_ptxas: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "pagedkv.h"))
    nv = nvcc()
    objs, cmds = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if force or verbose_ptxas or not _newer(o, [s] + headers):
            if src.endswith(".cpp"):      # host-only C++ (the block manager): the host compiler
                cmds.append([cxx(), "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-Wall",
                             "-I", os.path.join(ROOT, "include"), "-c", s, "-o", o])
            else:
                cmds.append([nv, *_flags(verbose_ptxas), "-c", s, "-o", o])
    if cmds:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(cmds), os.cpu_count() or 1)) as ex:
            futs = [ex.submit(subprocess.run, c, capture_output=True, text=True) for c in cmds]
            for c, fu in zip(cmds, futs):
                r = fu.result()
                if verbose_ptxas or r.returncode:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode:
                    raise RuntimeError(f"nvcc failed: {' '.join(c)}")
    if force or cmds or not _newer(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([nv, *ARCH, "-shared", "-o", tmp, *objs, "-lcuda"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
