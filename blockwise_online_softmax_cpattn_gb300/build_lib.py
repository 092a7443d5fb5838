"""Builds libcpattn.so in-tree with nvcc for sm_103a.

Each CUDA translation unit under csrc/ is compiled separately (in parallel) and
linked into ``blockwise_online_softmax_cpattn_gb300/libcpattn.so``.  The CUDA
runtime is linked statically; the tensor-map encoder is reached through the
runtime's driver entry point, so no libcuda link is needed at build time.

``build(debug=True)`` builds the same sources with CPATTN_DEBUG defined into
``libcpattn_debug.so``: the tensor-core kernels then check every computed tensor
row against its tensor's extent, latch CPATTN_ERR_BOUNDS and skip the access on
a failure.  The binding loads that library instead when the environment sets
CPATTN_DEBUG_LIB=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcpattn.so")
OBJ_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libcpattn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = [os.environ.get("NVCC", ""), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc") or ""]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _fingerprint(flags) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    h.update(" ".join(ARCH + flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Compile (if stale) and return the path of libcpattn.so (libcpattn_debug.so
    with debug=True)."""
    obj_dir, lib = (OBJ_DEBUG, LIB_DEBUG) if debug else (OBJ, LIB)
    flags = FLAGS + (["-DCPATTN_DEBUG"] if debug else [])
    stamp = os.path.join(obj_dir, "fingerprint")
    fp = _fingerprint(flags)
    if not force and not ptxas_info and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read() == fp:
                return lib
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(fp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
