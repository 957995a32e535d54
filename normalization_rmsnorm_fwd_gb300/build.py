"""Build ``libcrmsnorm.so`` in-tree with nvcc for sm_103a.

Every ``csrc/*.cu`` is compiled in parallel to an object file under
``_build/`` and the objects are linked into one shared library
(CUDA runtime linked statically).  A stamp of the sources and flags skips
the build when nothing changed.  Run ``python -m
normalization_rmsnorm_fwd_gb300.build [-v] [--debug]`` (``-v`` adds
``-Xptxas -v``; ``--debug`` builds ``_build_debug/libcrmsnorm_debug.so``
with ``-DCRMSN_DEBUG``: the kernels' bounds guard, read back with
``crmsn_debug_status``).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libcrmsnorm.so")
OUT_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(OUT_DEBUG, "libcrmsnorm_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden symbols: the shared library exports only the C ABI of crmsnorm.h,
# so its internal template statics (launch caches) are never merged with
# another library's in the same process.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcrmsnorm")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(extra) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    h.update(" ".join(NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DCRMSN_DEBUG"] if debug else [])
    out, lib = (OUT_DEBUG, LIB_DEBUG) if debug else (OUT, LIB)
    os.makedirs(out, exist_ok=True)
    stamp_path = os.path.join(out, "stamp")
    stamp = _stamp(extra)
    if (not force and os.path.exists(lib) and os.path.exists(stamp_path)
            and open(stamp_path).read() == stamp):
        return lib
    nvcc = _nvcc()
    srcs = _sources()
    objs = [os.path.join(out, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        for src, r in ex.map(compile_one, zip(srcs, objs)):
            if verbose or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
