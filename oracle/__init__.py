"""Q8_0 oracle: plain, slow CPU reference of the row quantizer and of qdot_t.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library in ``gemm_q8_qdot_gb300`` and the product
path never calls it.

The arithmetic lives in ``q8_oracle.c`` (plain C, compiled here with gcc, no
FMA contraction, no fast math).  This module only compiles it and marshals
numpy arrays.  What each function computes, and the passages of the Phobos
pages it follows, are stated in the C file:

* "Quantized built-ins and formats", section "Q8_0" -- block format and the
  qdot_t formula with the inner sum in integers;
* "Phobos Language Spec", section 10 "Quantized built-ins" -- operand shapes,
  the qmma_t scale layout [K/32, N];
* same spec, section 9, Elementwise table -- round() ties to even;
* same spec, section 10, Q5_0 row (q50_qdot_t) -- Q5_0 weight blocks (qh word,
  16 nibble bytes, elements q - 16) against Q8_0 activations.

Pins: every function here is checked against values fixed by the pages and by
mathematics (brute force in exact rationals, closed forms, invariants, a
float64 library matmul on dequantized values) in ``tests/test_oracle_pins.py``
and, for Q5_0, ``tests/test_oracle_q50_pins.py``.
The exact f32 bit pattern of qdot_t's output is not fixed by the pages (the
summation order and FMA contraction are free), so that is held to a tolerance,
not pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

QK = 32
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_libs: dict[tuple[int, bool], ctypes.CDLL] = {}
_lock = threading.Lock()

_I8P = ctypes.POINTER(ctypes.c_int8)
_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)
_I64P = ctypes.POINTER(ctypes.c_int64)
_I64 = ctypes.c_int64


def lib_path(mutant: int = 0, omp: bool = False) -> str:
    return os.path.join(_BUILD, f"liboracle_m{mutant}{'_omp' if omp else ''}.so")


def build(mutant: int = 0, force: bool = False, omp: bool = False) -> str:
    """Compile q8_oracle.c into a shared library (mutant 0 = the real oracle).

    omp=True builds the same source with -fopenmp: the loops over quantizer
    rows and output elements run on every host core, each row and element
    still computed by the single-thread build's sequential loop.
    """
    out = lib_path(mutant, omp)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    if omp:
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0, omp: bool = False) -> ctypes.CDLL:
    key = (mutant, omp)
    with _lock:
        if key not in _libs:
            lib = ctypes.CDLL(build(mutant, omp=omp))
            lib.oracle_quantize_q8_0.argtypes = [_F32P, _I8P, _F32P, _I64, _I64]
            lib.oracle_blocksums_q8_0.argtypes = [_I8P, _I8P, _I64P, _I64, _I64, _I64]
            lib.oracle_qdot_q8_0.argtypes = [_I8P, _F32P, _I8P, _F32P, _F64P, _F64P, _I64, _I64, _I64]
            lib.oracle_qdot_q8_0_ex.argtypes = [_I8P, _F32P, _I8P, _F32P, _F64P, _F64P,
                                                _I64, _I64, _I64, ctypes.c_int]
            _U8P = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_decode_q5_0.argtypes = [_U8P, _I8P, _I64, _I64]
            lib.oracle_blocksums_q5_0.argtypes = [_I8P, _U8P, _I64P, _I64, _I64, _I64]
            lib.oracle_qdot_q5_0.argtypes = [_I8P, _F32P, _U8P, _F32P, _F64P, _F64P,
                                             _I64, _I64, _I64, ctypes.c_int]
            for fn in ("oracle_quantize_q8_0", "oracle_blocksums_q8_0", "oracle_qdot_q8_0",
                       "oracle_qdot_q8_0_ex", "oracle_decode_q5_0", "oracle_blocksums_q5_0",
                       "oracle_qdot_q5_0"):
                getattr(lib, fn).restype = None
            lib.oracle_mutant.restype = ctypes.c_int
            lib.oracle_threads.restype = ctypes.c_int
            assert lib.oracle_mutant() == mutant
            _libs[key] = lib
        return _libs[key]


def threads(omp: bool = True) -> int:
    """Host threads the (omp) build's loops run on."""
    return int(_lib(0, omp).oracle_threads())


def _p(arr: np.ndarray, ctype):
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _c(arr, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(arr), dtype=dtype)


def quantize_q8_0(x, mutant: int = 0, omp: bool = False):
    """x f32 [R, K] -> (q int8 [R, K], s f32 [R, K/32])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    R, K = x.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    q = np.empty((R, K), np.int8)
    s = np.empty((R, K // QK), np.float32)
    _lib(mutant, omp).oracle_quantize_q8_0(_p(x, ctypes.c_float), _p(q, ctypes.c_int8),
                                      _p(s, ctypes.c_float), R, K)
    return q, s


def blocksums(a, w, mutant: int = 0, omp: bool = False) -> np.ndarray:
    """a int8 [M, K], w int8 [N, K] -> S int64 [M, N, K/32] (exact block sums)."""
    a = _c(a, np.int8)
    w = _c(w, np.int8)
    M, K = a.shape
    N, K2 = w.shape
    if K != K2 or K % QK:
        raise ValueError("shape mismatch")
    S = np.empty((M, N, K // QK), np.int64)
    _lib(mutant, omp).oracle_blocksums_q8_0(_p(a, ctypes.c_int8), _p(w, ctypes.c_int8),
                                       _p(S, ctypes.c_int64), M, N, K)
    return S


def qdot(a, a_scales, w, w_scales, ws_layout: int = 0, mutant: int = 0, omp: bool = False):
    """qdot_t in double: returns (out f64 [M, N], bound f64 [M, N]).

    ws_layout 0: w_scales [N, K/32] (qdot_t); 1: w_scales [K/32, N] (qmma_t).
    """
    a = _c(a, np.int8)
    w = _c(w, np.int8)
    a_scales = _c(a_scales, np.float32)
    w_scales = _c(w_scales, np.float32)
    M, K = a.shape
    N, K2 = w.shape
    KB = K // QK
    if K != K2 or K % QK or a_scales.shape != (M, KB):
        raise ValueError("shape mismatch")
    if w_scales.shape != ((N, KB) if ws_layout == 0 else (KB, N)):
        raise ValueError("w_scales shape mismatch")
    out = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    lib = _lib(mutant, omp)
    args = (_p(a, ctypes.c_int8), _p(a_scales, ctypes.c_float), _p(w, ctypes.c_int8),
            _p(w_scales, ctypes.c_float), _p(out, ctypes.c_double), _p(bound, ctypes.c_double),
            M, N, K)
    if ws_layout == 0:
        lib.oracle_qdot_q8_0(*args)
    else:
        lib.oracle_qdot_q8_0_ex(*args, int(ws_layout))
    return out, bound


# ---------------------------------------------------------------- Q5_0 weights

Q50_BYTES = 20  # bytes per 32-element Q5_0 block without its scale


def decode_q5_0(w5, K: int, mutant: int = 0, omp: bool = False) -> np.ndarray:
    """Q5_0 blocks uint8 [R, K/32 * 20] -> int8 [R, K] (q - 16)."""
    w5 = _c(w5, np.uint8)
    R = w5.shape[0]
    if K % QK or w5.shape[1] != K // QK * Q50_BYTES:
        raise ValueError("shape mismatch")
    w = np.empty((R, K), np.int8)
    _lib(mutant, omp).oracle_decode_q5_0(_p(w5, ctypes.c_uint8), _p(w, ctypes.c_int8), R, K)
    return w


def blocksums_q5_0(a, w5, mutant: int = 0, omp: bool = False) -> np.ndarray:
    """a int8 [M, K], Q5_0 blocks [N, K/32 * 20] -> S int64 [M, N, K/32]."""
    a = _c(a, np.int8)
    w5 = _c(w5, np.uint8)
    M, K = a.shape
    N = w5.shape[0]
    if K % QK or w5.shape[1] != K // QK * Q50_BYTES:
        raise ValueError("shape mismatch")
    S = np.empty((M, N, K // QK), np.int64)
    _lib(mutant, omp).oracle_blocksums_q5_0(_p(a, ctypes.c_int8), _p(w5, ctypes.c_uint8),
                                       _p(S, ctypes.c_int64), M, N, K)
    return S


def qdot_q5_0(a, a_scales, w5, w_scales, ws_layout: int = 0, mutant: int = 0, omp: bool = False):
    """q50_qdot_t (ws_layout 0) / q50_qmma_t scale layout (1) in double: (out, bound)."""
    a = _c(a, np.int8)
    w5 = _c(w5, np.uint8)
    a_scales = _c(a_scales, np.float32)
    w_scales = _c(w_scales, np.float32)
    M, K = a.shape
    N = w5.shape[0]
    KB = K // QK
    if K % QK or w5.shape[1] != KB * Q50_BYTES or a_scales.shape != (M, KB):
        raise ValueError("shape mismatch")
    if w_scales.shape != ((N, KB) if ws_layout == 0 else (KB, N)):
        raise ValueError("w_scales shape mismatch")
    out = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    _lib(mutant, omp).oracle_qdot_q5_0(_p(a, ctypes.c_int8), _p(a_scales, ctypes.c_float),
                                  _p(w5, ctypes.c_uint8), _p(w_scales, ctypes.c_float),
                                  _p(out, ctypes.c_double), _p(bound, ctypes.c_double),
                                  M, N, K, int(ws_layout))
    return out, bound
