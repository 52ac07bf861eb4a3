"""ORACLE -- test infrastructure only.

Python access to the plain C oracle (``oracle.c``) of the FP4 weight-only (W4A16) linear
layer.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product package never does.

Every function here only marshals numpy arrays to the C code; the arithmetic, with its
citations, is in ``oracle.c``.  bf16 tensors are numpy ``uint16`` arrays of bit patterns.
Formats: ``NVFP4 = 0`` (E2M1 codes, E4M3 scale per 16, fp32 global multiplier) and
``MXFP4 = 1`` (E2M1 codes, E8M0 scale per 32, no global).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

NVFP4, MXFP4 = 0, 1
GROUP = {NVFP4: 16, MXFP4: 32}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-pthread", "-o", _SO, _SRC, "-lm"]
        subprocess.check_call(cmd)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.orc_e2m1_value.argtypes = [ctypes.c_uint]
        lib.orc_e2m1_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e8m0_value.argtypes = [ctypes.c_uint]
        lib.orc_e8m0_value.restype = ctypes.c_double
        lib.orc_e2m1_from_real.argtypes = [ctypes.c_double]
        lib.orc_e2m1_from_real.restype = ctypes.c_uint
        lib.orc_e4m3_from_real.argtypes = [ctypes.c_double]
        lib.orc_e4m3_from_real.restype = ctypes.c_uint
        lib.orc_mx_exponent.argtypes = [ctypes.c_double]
        lib.orc_mx_exponent.restype = ctypes.c_int
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_quantize_nvfp4.argtypes = [_P, _I64, _I64, _P, _P, _P, ctypes.c_int]
        lib.orc_quantize_nvfp4.restype = ctypes.c_int
        lib.orc_quantize_mxfp4.argtypes = [_P, _I64, _I64, _P, _P, ctypes.c_int]
        lib.orc_quantize_mxfp4.restype = ctypes.c_int
        lib.orc_dequant.argtypes = [ctypes.c_int, _P, _P, ctypes.c_float, _I64, _I64, _P,
                                    ctypes.c_int]
        lib.orc_dequant.restype = ctypes.c_int
        lib.orc_gemm.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, _P, ctypes.c_float, _I64,
                                 _P, _I64, _P, _P, _P, ctypes.c_int]
        lib.orc_gemm.restype = ctypes.c_int
        lib.orc_greedy.argtypes = [_P, _I64, _I64, _P, _P]
        lib.orc_greedy.restype = ctypes.c_int
        lib.orc_silu_mul.argtypes = [_P, _I64, _I64, _P]
        lib.orc_silu_mul.restype = ctypes.c_int
        lib.orc_quantize_act.argtypes = [ctypes.c_int, _P, _I64, _I64, ctypes.c_float, _P, _P,
                                         _P, ctypes.c_int]
        lib.orc_quantize_act.restype = ctypes.c_int
        lib.orc_gemm_w4a4.argtypes = [ctypes.c_int, _P, _I64, _I64, ctypes.c_float, _P, _P,
                                      ctypes.c_float, _I64, _P, _I64, _P, _P, _P, ctypes.c_int]
        lib.orc_gemm_w4a4.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    return max(1, min(256, os.cpu_count() or 1))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ----------------------------------------------------------------- format decoders
def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(byte)


def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(byte)


def e2m1_from_real(q: float) -> int:
    return _load().orc_e2m1_from_real(q)


def e4m3_from_real(x: float) -> int:
    return _load().orc_e4m3_from_real(x)


def mx_exponent(amax: float) -> int:
    return _load().orc_mx_exponent(amax)


def f32_to_bf16(x: float) -> int:
    return _load().orc_f32_to_bf16(x)


# ---------------------------------------------------------------------- quantisers
def quantize_nvfp4(W: np.ndarray, nthreads: int | None = None):
    """W: bf16 bits [N, K] -> (codes u8 [N, K/2], scales u8 [N, K/16], global float)."""
    W, wp = _c(W, np.uint16)
    N, K = W.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    g = ctypes.c_float(0.0)
    rc = _load().orc_quantize_nvfp4(wp, N, K, codes.ctypes.data, scales.ctypes.data,
                                    ctypes.addressof(g), nthreads or threads())
    if rc:
        raise ValueError("orc_quantize_nvfp4 rejected the input")
    return codes, scales, float(g.value)


def quantize_mxfp4(W: np.ndarray, nthreads: int | None = None):
    """W: bf16 bits [N, K] -> (codes u8 [N, K/2], scales u8 [N, K/32])."""
    W, wp = _c(W, np.uint16)
    N, K = W.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 32), np.uint8)
    rc = _load().orc_quantize_mxfp4(wp, N, K, codes.ctypes.data, scales.ctypes.data,
                                    nthreads or threads())
    if rc:
        raise ValueError("orc_quantize_mxfp4 rejected the input")
    return codes, scales


def quantize(fmt: int, W: np.ndarray):
    """(codes, scales, global) for either format; MXFP4's global is 1.0."""
    if fmt == NVFP4:
        return quantize_nvfp4(W)
    c, s = quantize_mxfp4(W)
    return c, s, 1.0


# ---------------------------------------------------------------- dequant and GEMM
def dequant(fmt: int, codes, scales, G: float, N: int, K: int) -> np.ndarray:
    """w[n][k] in fp32 as the layer uses it."""
    codes, cp = _c(codes, np.uint8)
    scales, sp = _c(scales, np.uint8)
    out = np.empty((N, K), np.float32)
    if _load().orc_dequant(fmt, cp, sp, G, N, K, out.ctypes.data, threads()):
        raise ValueError("orc_dequant rejected the input")
    return out


def gemm(fmt: int, A, codes, scales, G: float, N: int, cols=None, want_f64: bool = False,
         nthreads: int | None = None):
    """y = A . W^T.  A: bf16 bits [M, K].  Returns (y fp32 [M, n], y_bf16 bits [M, n]) and,
    if ``want_f64``, the fp64-accumulated sums as a third element.  ``cols`` restricts the
    output to those columns n (in the given order); ``nthreads`` (default: every core) splits
    the output columns between threads, which changes no result bit."""
    A, ap = _c(A, np.uint16)
    codes, cp = _c(codes, np.uint8)
    scales, sp = _c(scales, np.uint8)
    M, K = A.shape
    if cols is None:
        ncols, colp, keep = N, None, None
    else:
        keep = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        ncols, colp = keep.size, keep.ctypes.data
    y = np.empty((M, ncols), np.float32)
    ybf = np.empty((M, ncols), np.uint16)
    y64 = np.empty((M, ncols), np.float64) if want_f64 else None
    rc = _load().orc_gemm(fmt, ap, M, K, cp, sp, G, N, colp, ncols, y.ctypes.data,
                          y64.ctypes.data if want_f64 else None, ybf.ctypes.data,
                          nthreads or threads())
    if rc:
        raise ValueError("orc_gemm rejected the input")
    return (y, ybf, y64) if want_f64 else (y, ybf)


def quantize_act(fmt: int, A, alpha: float = 1.0):
    """W4A4 activation quantiser (decisions in fp32).  A: bf16 bits [M, K] ->
    (codes u8 [M, K/2], scales u8 [M, K/g], dequantised activations fp32 [M, K])."""
    A, ap = _c(A, np.uint16)
    M, K = A.shape
    g = 16 if fmt == NVFP4 else 32
    codes = np.empty((M, K // 2), np.uint8)
    scales = np.empty((M, K // g), np.uint8)
    aq = np.empty((M, K), np.float32)
    if _load().orc_quantize_act(fmt, ap, M, K, alpha, codes.ctypes.data, scales.ctypes.data,
                                aq.ctypes.data, threads()):
        raise ValueError("orc_quantize_act rejected the input")
    return codes, scales, aq


def gemm_w4a4(fmt: int, A, alpha: float, codes, scales, G: float, N: int, cols=None,
              want_f64: bool = False):
    """The W4A4 layer: the activations A (bf16 bits [M, K]) quantised by quantize_act with
    the activation global ``alpha``, then the same fp32 GEMM as ``gemm``."""
    A, ap = _c(A, np.uint16)
    codes, cp = _c(codes, np.uint8)
    scales, sp = _c(scales, np.uint8)
    M, K = A.shape
    if cols is None:
        ncols, colp, keep = N, None, None
    else:
        keep = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        ncols, colp = keep.size, keep.ctypes.data
    y = np.empty((M, ncols), np.float32)
    ybf = np.empty((M, ncols), np.uint16)
    y64 = np.empty((M, ncols), np.float64) if want_f64 else None
    rc = _load().orc_gemm_w4a4(fmt, ap, M, K, alpha, cp, sp, G, N, colp, ncols,
                               y.ctypes.data, y64.ctypes.data if want_f64 else None,
                               ybf.ctypes.data, threads())
    if rc:
        raise ValueError("orc_gemm_w4a4 rejected the input")
    return (y, ybf, y64) if want_f64 else (y, ybf)


def greedy(ybf):
    """Greedy choice per row of bf16 outputs [M, N] (bits): (index int32 [M], value bits
    uint16 [M]); the largest value, ties to the lowest index, NaN above every number."""
    ybf, yp = _c(ybf, np.uint16)
    M, N = ybf.shape
    idx = np.empty(M, np.int32)
    val = np.empty(M, np.uint16)
    if _load().orc_greedy(yp, M, N, idx.ctypes.data, val.ctypes.data):
        raise ValueError("orc_greedy rejected the input")
    return idx, val


def silu_mul(y):
    """SiLU-gated MLP input from fused gate_up sums y fp32 [M, 2I]: bf16 bits [M, I] of
    silu(gate) * up, evaluated in fp64 and rounded once."""
    y, yp = _c(y, np.float32)
    M, N2 = y.shape
    if N2 % 2:
        raise ValueError("a fused gate_up output has an even number of columns")
    out = np.empty((M, N2 // 2), np.uint16)
    if _load().orc_silu_mul(yp, M, N2 // 2, out.ctypes.data):
        raise ValueError("orc_silu_mul rejected the input")
    return out


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32)
