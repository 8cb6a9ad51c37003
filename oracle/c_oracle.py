"""The plain C statement of the W4A16 layer (``w4_oracle_c.c``), built with gcc
and called through ctypes. TEST INFRASTRUCTURE ONLY (see the package
docstring): bench.py times it as the CPU baseline, and the tests pin it to the
numpy oracle. It shares no code with the CUDA path."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "w4_oracle_c.c")
_LIB = os.path.join(_DIR, "_build", "libw4oracle.so")
_lib = None


def build() -> str:
    """Compile ``w4_oracle_c.c`` (gcc -O3, pthreads; no machine-specific flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.run(["gcc", "-O3", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        fn = lib.w4o_w4a16_linear
        fn.restype = ctypes.c_int
        P, I64 = ctypes.c_void_p, ctypes.c_int64
        fn.argtypes = [P, I64, I64, P, I64, P, ctypes.c_int, P, I64, P, P, ctypes.c_int]
        _lib = lib
    return _lib


def threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def w4a16_linear(x_bits, qweight, w_scale, group, zeros_bits=None, bias_bits=None, scale_dtype="f16",
                 nthreads=None) -> np.ndarray:
    """Same arguments and result as the numpy oracle's ``w4a16_linear``
    (float32 ``[M, N]`` before the bf16 cast), computed by the C code."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    qw = np.ascontiguousarray(qweight, dtype=np.int32)
    if scale_dtype == "f16":
        s = np.ascontiguousarray(np.asarray(w_scale, dtype=np.float16)).view(np.uint16)
    elif scale_dtype == "bf16":
        s = np.ascontiguousarray(w_scale, dtype=np.uint16)
    else:
        raise ValueError(scale_dtype)
    z = None if zeros_bits is None else np.ascontiguousarray(zeros_bits, dtype=np.uint16)
    b = None if bias_bits is None else np.ascontiguousarray(bias_bits, dtype=np.uint16)
    M, K = x.shape
    N = qw.shape[1]
    out = np.empty((M, N), dtype=np.float32)
    rc = _load().w4o_w4a16_linear(x.ctypes.data, M, K, qw.ctypes.data, N, s.ctypes.data,
                                  1 if scale_dtype == "bf16" else 0, None if z is None else z.ctypes.data, group,
                                  None if b is None else b.ctypes.data, out.ctypes.data,
                                  threads() if nthreads is None else nthreads)
    if rc != 0:
        raise RuntimeError(f"w4o_w4a16_linear failed ({rc})")
    return out
