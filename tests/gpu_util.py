"""Shared helpers of the GPU parity tests (test plumbing, no method arithmetic)."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def lib():
    from bit_kv_cache_keyquant_gb300 import build
    build.build()
    from bit_kv_cache_keyquant_gb300 import kvq
    return kvq


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


_curand = None


def curand_philox():
    """ctypes handle of tests/curand_philox_ref.cu compiled for sm_103a."""
    global _curand
    if _curand is None:
        d = tempfile.mkdtemp(prefix="kvq_curand_")
        so = os.path.join(d, "libcurand_ref.so")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler",
                        "-fPIC", os.path.join(HERE, "curand_philox_ref.cu"), "-o", so], check=True)
        _curand = ctypes.CDLL(so)
        _curand.curand_philox_ref.restype = ctypes.c_int
        _curand.curand_philox_ref.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p]
    return _curand


def attn_tol(want):
    """Per-element tolerance of an fp16 attention output against the binary64
    oracle: max-abs 2e-3, widened to one fp16 ulp of the oracle value where the
    fp16 output grid itself is coarser than 2e-3 (|o| >= 4)."""
    w = np.abs(np.asarray(want, np.float64))
    ulp = np.spacing(w.astype(np.float16)).astype(np.float64)
    return np.maximum(2e-3, ulp)


def assert_attn_close(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), what
    err = np.abs(got - want)
    tol = attn_tol(want)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, worst {err.max():.3e} " \
                          f"(|o| there {np.abs(want).flat[err.argmax()]:.3f})"
