"""ctypes loader for the C++ oracle (ref_cpu.cpp) and its build step.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's
CPU-baseline leg. See ref_cpu.cpp for what it computes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .ref import OracleError

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_cpu.cpp")
_LIB = os.path.join(_HERE, "liboracle_subm3d.so")
_lib = None

_ERRORS = {-1: "bad argument", -2: "coordinate outside the grid", -3: "duplicate coordinate"}


def build(force: bool = False) -> str:
    """Compile ref_cpu.cpp into liboracle_subm3d.so (g++ -O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c++17",
                        _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_threads.argtypes = [ctypes.c_int]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_kernel_map.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_void_p, ctypes.c_int, i64p]
        lib.oracle_kernel_map.restype = ctypes.c_int
        lib.oracle_forward_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int, i64p]
        lib.oracle_forward_rows.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads(nthreads: int = 0) -> int:
    """OpenMP thread count the oracle calls use (nthreads <= 0: OpenMP default)."""
    return _load().oracle_threads(nthreads)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def _raise(rc, bad):
    raise OracleError(f"oracle: {_ERRORS.get(rc, rc)} (row {bad})")


def kernel_map(coords, res, nthreads: int = 0) -> np.ndarray:
    """nbr int32 [N, 27] (same definition as ref.kernel_map)."""
    c = np.ascontiguousarray(coords, dtype=np.int32)
    N = c.shape[0]
    nbr = np.empty((N, 27), dtype=np.int32)
    bad = ctypes.c_int64(-1)
    rc = _load().oracle_kernel_map(_ptr(c), N, int(res), _ptr(nbr), nthreads, ctypes.byref(bad))
    if rc:
        _raise(rc, bad.value)
    return nbr


def forward_rows(coords, feats, weight, bias, res, rows=None, nthreads: int = 0) -> np.ndarray:
    """Output rows (all if rows is None) as float64 [len(rows), O] (same definition as
    ref.subm_conv3d_rows), from float32 inputs accumulated in double."""
    c = np.ascontiguousarray(coords, dtype=np.int32)
    f = np.ascontiguousarray(feats, dtype=np.float32)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    N, I = f.shape
    O = w.shape[0]
    if c.shape[0] != N or w.shape[1:] != (3, 3, 3, I):
        raise OracleError("shape mismatch")
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    r = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    out = np.empty((r.shape[0], O), dtype=np.float64)
    bad = ctypes.c_int64(-1)
    rc = _load().oracle_forward_rows(_ptr(c), N, int(res), _ptr(f), I, _ptr(w), O, _ptr(b),
                                     _ptr(r), r.shape[0], _ptr(out), nthreads, ctypes.byref(bad))
    if rc:
        _raise(rc, bad.value)
    return out
