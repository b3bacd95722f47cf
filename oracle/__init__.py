"""CPU oracle for D = A * B^T (fp16 in, double accumulate, one fp16 rounding).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The CUDA library never links, loads or calls it, and it never
imports the CUDA library: the two meet only through the seeded fp16 bit
patterns both are given.

The arithmetic lives in ``gemm_oracle.c`` (plain C loops, see its header for
the definition and the passages it follows).  This module builds that file
with gcc into ``oracle/_build/`` and exposes it through ctypes:

* ``half_to_double(bits)`` / ``double_to_half(values)`` -- the converters,
  written from the IEEE 754 binary16 definition.
* ``gemm_tn(a_bits, b_bits, threads)`` -- the full M x N product.
* ``gemm_tn_sampled(a_bits, b_bits, rows, cols)`` -- selected elements.
* ``gemm_tn_f16acc(a_bits, b_bits)`` -- the product with an fp16 accumulator
  rounded after every 16-deep K slice (the page's MMA atom).
* ``gemm_scaled(a_bits, b_bits, c_bits, alpha, beta, b_kn)`` -- the scaled
  form alpha * A op(B) + beta * C, with B N x K (TN) or K x N (NN).
* ``minimum_stages(copy, compute)`` -- S_min = ceil(copy/compute) + 1
  ("第 6 课：Shared Memory 布局与异步流水", section 4).

Parity status of each function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c with gcc (no -ffast-math, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    i64, u16p = ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_gemm_tn.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int]
    lib.oracle_gemm_tn.restype = ctypes.c_int
    lib.oracle_gemm_tn_sampled.argtypes = [u16p, u16p, i64, i64, i64, i64p, i64p, i64, u16p]
    lib.oracle_gemm_tn_sampled.restype = ctypes.c_int
    lib.oracle_gemm_scaled.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_int, ctypes.c_int]
    lib.oracle_gemm_scaled.restype = ctypes.c_int
    lib.oracle_gemm_tn_f16acc.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int]
    lib.oracle_gemm_tn_f16acc.restype = ctypes.c_int
    lib.oracle_minimum_stages.argtypes = [i64, i64]
    lib.oracle_minimum_stages.restype = ctypes.c_int64
    return lib


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIBRARY points the loader at an edited build of gemm_oracle.c;
        # the mutation tests use it to check that the pins reject planted mistakes.
        path = os.environ.get("ORACLE_LIBRARY") or build()
        _lib = _bind(ctypes.CDLL(path))
    return _lib


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of gemm_oracle.c to `out_path` (used by the
    mutation tests to plant a mistake in the oracle)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", out_path, src, "-lpthread", "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are fp16 bit patterns (uint16 or float16 arrays)")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def half_to_double(bits, lib=None) -> np.ndarray:
    lib = lib or _load()
    b = _u16(np.asarray(bits)).ravel()
    return np.array([lib.oracle_half_to_double(int(x)) for x in b], dtype=np.float64)


def double_to_half(values, lib=None) -> np.ndarray:
    lib = lib or _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib.oracle_double_to_half(float(x)) for x in v], dtype=np.uint16)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def gemm_tn(a_bits: np.ndarray, b_bits: np.ndarray, threads: int | None = None, lib=None) -> np.ndarray:
    """D (M x N, fp16 bits as uint16) for A (M x K) and B (N x K) fp16 bits."""
    a, b = _u16(a_bits), _u16(b_bits)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("A must be M x K and B N x K")
    M, K = a.shape
    N = b.shape[0]
    d = np.zeros((M, N), dtype=np.uint16)
    rc = (lib or _load()).oracle_gemm_tn(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                _ptr(d, ctypes.c_uint16), M, N, K, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_tn rejected its arguments")
    return d


def gemm_tn_f16acc(a_bits: np.ndarray, b_bits: np.ndarray, threads: int | None = None,
                   lib=None) -> np.ndarray:
    """D = A B^T with an fp16 accumulator rounded after every 16-deep K slice."""
    a, b = _u16(a_bits), _u16(b_bits)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("A must be M x K and B N x K")
    M, K = a.shape
    N = b.shape[0]
    d = np.zeros((M, N), dtype=np.uint16)
    rc = (lib or _load()).oracle_gemm_tn_f16acc(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                               _ptr(d, ctypes.c_uint16), M, N, K,
                                               threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_tn_f16acc rejected its arguments")
    return d


def gemm_scaled(a_bits: np.ndarray, b_bits: np.ndarray, c_bits, alpha: float, beta: float,
                b_kn: bool, threads: int | None = None, lib=None) -> np.ndarray:
    """D = fp16(alpha * A op(B) + beta * C): B is K x N when b_kn, else N x K.
    C (M x N fp16 bits) is not read when beta == 0 and may then be None."""
    a, b = _u16(a_bits), _u16(b_bits)
    M, K = a.shape
    if b_kn:
        if b.shape[0] != K:
            raise ValueError("B must be K x N")
        N = b.shape[1]
    else:
        if b.shape[1] != K:
            raise ValueError("B must be N x K")
        N = b.shape[0]
    c = None
    if c_bits is not None:
        c = _u16(c_bits)
        if c.shape != (M, N):
            raise ValueError("C must be M x N")
    d = np.zeros((M, N), dtype=np.uint16)
    c_ptr = _ptr(c, ctypes.c_uint16) if c is not None else None
    rc = (lib or _load()).oracle_gemm_scaled(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                            c_ptr, _ptr(d, ctypes.c_uint16), M, N, K,
                                            float(alpha), float(beta), 1 if b_kn else 0,
                                            threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_scaled rejected its arguments")
    return d


def gemm_tn_sampled(a_bits: np.ndarray, b_bits: np.ndarray, rows, cols, lib=None) -> np.ndarray:
    """D[rows[s], cols[s]] (fp16 bits) for each sample s."""
    a, b = _u16(a_bits), _u16(b_bits)
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols must have one shape")
    out = np.zeros(r.shape, dtype=np.uint16)
    rc = (lib or _load()).oracle_gemm_tn_sampled(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                        M, N, K, _ptr(r, ctypes.c_int64), _ptr(c, ctypes.c_int64),
                                        r.size, _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_gemm_tn_sampled rejected its arguments")
    return out


def minimum_stages(copy_cycles: int, compute_cycles: int, lib=None) -> int:
    return int((lib or _load()).oracle_minimum_stages(int(copy_cycles), int(compute_cycles)))
