"""Seeded synthetic inputs (bf16 normal tensors) shared by the oracle and the GPU path.

Holds none of the FP4 layer's arithmetic: it only draws N(0, sigma) values with a
counter-based generator (SplitMix64 + Box-Muller, see ``synth.c``) so that any row of
any tensor can be regenerated on its own.  Tensors are returned as numpy ``uint16``
arrays holding bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libvtsynth.so")
_lib = None

# Tensor ids used by the workloads: one id per (workload, layer, role) so that every
# weight and activation tensor is an independent stream.
ROLE_W, ROLE_A = 1, 2
ROLE_GATE, ROLE_UP, ROLE_DOWN, ROLE_O = 11, 12, 13, 14


def tensor_id(workload: int, layer: int, role: int, extra: int = 0) -> int:
    return (workload << 40) | (layer << 24) | (role << 8) | extra


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
               "-o", _SO, _SRC, "-lm"]
        subprocess.check_call(cmd)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_int]
        lib.synth_normal_bf16.restype = None
        lib.synth_normal_bf16_rows.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal_bf16_rows.restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, tid: int, sigma: float, rows: int, cols: int) -> np.ndarray:
    """bf16 bit patterns of a [rows, cols] tensor drawn from N(0, sigma^2)."""
    out = np.empty((rows, cols), dtype=np.uint16)
    if out.size:
        _load().synth_normal_bf16(seed, tid, sigma, rows, cols, out.ctypes.data, _threads())
    return out


def normal_bf16_rows(seed: int, tid: int, sigma: float, cols: int, row_idx) -> np.ndarray:
    """Rows ``row_idx`` of the same [*, cols] tensor, regenerated independently."""
    idx = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
    out = np.empty((idx.size, cols), dtype=np.uint16)
    if out.size:
        _load().synth_normal_bf16_rows(seed, tid, sigma, cols, idx.ctypes.data, idx.size,
                                       out.ctypes.data, _threads())
    return out


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 values (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)
