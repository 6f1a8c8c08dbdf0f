"""In-tree build of libgbattn.so with nvcc for sm_103a.

The library is compiled from csrc/*.cu into _lib/libgbattn.so next to this
file (git-ignored).  Translation units compile in parallel; a rebuild happens
only when a source or header is newer than the library or the library was
built for another host architecture.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libgbattn.so")
STAMP = os.path.join(LIBDIR, "host_arch.txt")
SOURCES = ["attn_api.cu", "prefill_sm103.cu", "decode_sm103.cu", "decode_pair_sm103.cu", "gemm_sm103.cu"]
HEADERS = [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "philox.cuh"),
           os.path.join(ROOT, "include", "gbattn.h"), os.path.join(ROOT, "include", "gbgemm.h"),
           os.path.join(ROOT, "include", "gblayer.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                           "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgbattn.so")


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        if f.read().strip() != platform.machine():
            return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libgbattn.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    objs = [os.path.join(LIBDIR, s.replace(".cu", ".o")) for s in SOURCES]

    def compile_one(i):
        cmd = [cc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, SOURCES[i]), "-o", objs[i]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (SOURCES[i], r.stdout, r.stderr))
        if verbose:
            print(r.stdout + r.stderr)

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        list(ex.map(compile_one, range(len(SOURCES))))
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH_FLAGS + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(platform.machine())
    for o in objs:
        os.remove(o)
    return LIB
