"""Build libkvq.so (the sm_103a CUDA library) in-tree with nvcc.

Each translation unit is compiled in parallel, then linked with the static
CUDA runtime into bit_kv_cache_keyquant_gb300/libkvq.so.  Rebuilds only
when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", f"-I{os.path.join(ROOT, 'include')}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the kvq CUDA library cannot be built")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "kvq.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    return _build_into(BUILD, LIB, [], verbose, ptxas_info)


def build_test_lib(out_dir: str) -> str:
    """A separate copy of the library for the tests of the failure paths only: built with
    KVQ_FAULT_INJECT, which adds the kvq_test_inject_wait hook (a KIVI decode stage left unfilled,
    shortened wait limits).  The product library (build()) never defines it."""
    os.makedirs(out_dir, exist_ok=True)
    return _build_into(os.path.join(out_dir, "obj"), os.path.join(out_dir, "libkvq_test.so"),
                       ["-DKVQ_FAULT_INJECT"], False, False)


def _build_into(obj_dir: str, lib: str, defines, verbose: bool, ptxas_info: bool) -> str:
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + list(defines)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                print(err)
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
