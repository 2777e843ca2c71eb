"""CPU oracle, in fp64 rounded once to fp16, for C = epilogue(A.B + bias)
(gemm_oracle.cpp) and for attention O = softmax(scale Q K^T) V
(attn_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg are the only callers.  The product library never imports this
package, and this package never imports the product.

The arithmetic lives in ``gemm_oracle.cpp`` (plain C++, no CUDA); this module
only builds it with g++ and marshals numpy arrays through ctypes.  Every
function states the passage it follows in the C++ file's header:
"writing-tilelang-kernels" (Kernel Anatomy, GEMM (Minimal), Pre-flight
Checklist) and "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels
from Python" (What you'll see, Why tile-level control matters).

Pins (tests/test_oracle_pins.py): exhaustive fp16 round trips and numpy's
float16 conversion for the rounding; a numerical integral of the normal
density for GELU; closed forms (identity, permutation, rank-1, zero K tail,
integer inputs) and a brute-force Python triple loop for the GEMM.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

EPI_NONE, EPI_BIAS, EPI_BIAS_RELU, EPI_BIAS_GELU_ERF, EPI_BIAS_SIGMOID, EPI_BIAS_GELU_TANH = 0, 1, 2, 3, 4, 5
EPILOGUES = {"none": EPI_NONE, "bias": EPI_BIAS, "bias_relu": EPI_BIAS_RELU,
             "bias_gelu_erf": EPI_BIAS_GELU_ERF, "bias_sigmoid": EPI_BIAS_SIGMOID,
             "bias_gelu_tanh": EPI_BIAS_GELU_TANH}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "gemm_oracle.cpp"), os.path.join(_HERE, "attn_oracle.cpp")]
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (portable flags: runs on x86-64 and aarch64)."""
    if not force and os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                           "-fno-fast-math", "-ffp-contract=off", *_SRCS, "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_epilogue.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_epilogue.restype = ctypes.c_double
    lib.oracle_half_to_double_n.argtypes = [u16p, i64, f64p]
    lib.oracle_double_to_half_n.argtypes = [f64p, i64, u16p]
    lib.oracle_gemm_rows.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                     i64p, i64, u16p, f64p, ctypes.c_int]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_gemm_elems.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                      i64p, i64p, i64, u16p, f64p, ctypes.c_int]
    lib.oracle_gemm_elems.restype = ctypes.c_int
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                                     i64p, i64, u16p, f64p, ctypes.c_int]
    lib.oracle_attn_rows.restype = ctypes.c_int
    _lib = lib
    return lib


def _p(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def _bits(x):
    """fp16 array (or its uint16 bit pattern) -> contiguous uint16 view."""
    if x is None:
        return None
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"oracle wants fp16 or uint16 bits, got {x.dtype}")
    return x


def _epi(epilogue):
    return EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)


def half_to_double(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(b.size, np.float64)
    _load().oracle_half_to_double_n(_p(b, ctypes.c_uint16), b.size, _p(out, ctypes.c_double))
    return out.reshape(np.shape(bits))


def double_to_half(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp16 bit patterns, round to nearest even (the oracle's own code)."""
    a = np.ascontiguousarray(x, dtype=np.float64).ravel()
    out = np.empty(a.size, np.uint16)
    _load().oracle_double_to_half_n(_p(a, ctypes.c_double), a.size, _p(out, ctypes.c_uint16))
    return out.reshape(np.shape(x))


def epilogue_scalar(x: float, epilogue) -> float:
    return _load().oracle_epilogue(float(x), _epi(epilogue))


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def gemm_rows(A, B, bias, epilogue, rows, threads: int = 0, want_f64: bool = False):
    """Rows `rows` of C (fp16 array [len(rows), N]); optionally y before rounding."""
    A, B, bias = _bits(A), _bits(B), _bits(bias)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, N), np.uint16)
    f64 = np.empty((rows.size, N), np.float64) if want_f64 else None
    rc = _load().oracle_gemm_rows(_p(A, ctypes.c_uint16), _p(B, ctypes.c_uint16),
                                  _p(bias, ctypes.c_uint16), M, N, K, _epi(epilogue),
                                  _p(rows, ctypes.c_int64), rows.size,
                                  _p(out, ctypes.c_uint16), _p(f64, ctypes.c_double), threads)
    if rc != 0:
        raise ValueError("oracle_gemm_rows: bad arguments")
    out = out.view(np.float16)
    return (out, f64) if want_f64 else out


def gemm(A, B, bias, epilogue, threads: int = 0, want_f64: bool = False):
    """The whole of C (fp16 [M, N])."""
    return gemm_rows(A, B, bias, epilogue, np.arange(np.shape(A)[0]), threads, want_f64)


def gemm_elems(A, B, bias, epilogue, ii, jj, threads: int = 0, want_f64: bool = False):
    """Elements C[ii[e], jj[e]] (fp16 vector)."""
    A, B, bias = _bits(A), _bits(B), _bits(bias)
    M, K = A.shape
    _, N = B.shape
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    assert ii.shape == jj.shape
    out = np.empty(ii.size, np.uint16)
    f64 = np.empty(ii.size, np.float64) if want_f64 else None
    rc = _load().oracle_gemm_elems(_p(A, ctypes.c_uint16), _p(B, ctypes.c_uint16),
                                   _p(bias, ctypes.c_uint16), M, N, K, _epi(epilogue),
                                   _p(ii, ctypes.c_int64), _p(jj, ctypes.c_int64), ii.size,
                                   _p(out, ctypes.c_uint16), _p(f64, ctypes.c_double), threads)
    if rc != 0:
        raise ValueError("oracle_gemm_elems: bad arguments")
    out = out.view(np.float16)
    return (out, f64) if want_f64 else out


def gemm_grouped(problems, epilogue, threads: int = 0):
    """Grouped GEMM ("grouped GEMM" in the tilelang documentation's advanced
    examples: many independent GEMMs in one launch).  By definition each
    problem's C_g = epilogue(A_g . B_g + bias_g) on its own, so this is `gemm`
    applied to every (A_g, B_g, bias_g) of `problems` in turn; an empty
    problem (M or N of 0) gives an empty C_g."""
    out = []
    for A, B, bias in problems:
        M, N = np.shape(A)[0], np.shape(B)[1]
        if M == 0 or N == 0:
            out.append(np.zeros((M, N), np.float16))
        else:
            out.append(gemm(A, B, bias if _epi(epilogue) != 0 else None, epilogue, threads))
    return out


def attention_rows(Q, K, V, causal, scale, rows, threads: int = 0, want_f64: bool = False):
    """Rows of O = softmax(scale Q K^T) V (attn_oracle.cpp) for (B, H, S, D)
    fp16 Q, K, V: `rows` index the flattened (B * H * S) query rows; returns
    an fp16 array [len(rows), D] (and the values before rounding)."""
    Q, K, V = _bits(Q), _bits(K), _bits(V)
    B, H, S, D = Q.shape
    assert K.shape == Q.shape and V.shape == Q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, D), np.uint16)
    f64 = np.empty((rows.size, D), np.float64) if want_f64 else None
    rc = _load().oracle_attn_rows(_p(Q, ctypes.c_uint16), _p(K, ctypes.c_uint16), _p(V, ctypes.c_uint16),
                                  B, H, S, D, 1 if causal else 0, float(scale), _p(rows, ctypes.c_int64), rows.size,
                                  _p(out, ctypes.c_uint16), _p(f64, ctypes.c_double), threads)
    if rc != 0:
        raise ValueError("oracle_attn_rows: bad arguments")
    out = out.view(np.float16)
    return (out, f64) if want_f64 else out


def attention(Q, K, V, causal, scale=None, threads: int = 0, want_f64: bool = False):
    """The whole of O (fp16, shape of Q).  scale defaults to 1/sqrt(D), the
    default of the scaled-dot-product attention the pages validate against."""
    B, H, S, D = np.shape(Q)
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    r = attention_rows(Q, K, V, causal, scale, np.arange(B * H * S), threads, want_f64)
    if want_f64:
        return r[0].reshape(B, H, S, D), r[1].reshape(B, H, S, D)
    return r.reshape(B, H, S, D)
