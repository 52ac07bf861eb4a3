"""ctypes declarations of the C ABI in include/vt_fp4.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvtfp4.so")

VT_OK, VT_ERR_INVALID_ARG, VT_ERR_UNSUPPORTED, VT_ERR_MISALIGNED, VT_ERR_CUDA, VT_ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "VT_OK", 1: "VT_ERR_INVALID_ARG", 2: "VT_ERR_UNSUPPORTED",
                3: "VT_ERR_MISALIGNED", 4: "VT_ERR_CUDA", 5: "VT_ERR_TIMEOUT"}

# Every symbol the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_ST = ctypes.c_int


class LaunchInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("grid", ctypes.c_int), ("warps_per_cta", ctypes.c_int),
                ("m_tile", ctypes.c_int), ("items", ctypes.c_int64),
                ("launches", ctypes.c_int64), ("calls", ctypes.c_int64),
                ("tile_epilogue", ctypes.c_int), ("stage_k_tiles", ctypes.c_int)]


class GemmOpts(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int), ("warps", ctypes.c_int), ("stages", ctypes.c_int),
                ("force_path", ctypes.c_int), ("wait_limit_us", ctypes.c_int),
                ("withhold_weights", ctypes.c_int)]


SIGNATURES = {
    "vt_fp4_prepack_bytes": (_ST, [ctypes.c_int, _I64, _I64, ctypes.POINTER(_SZ)]),
    "vt_fp4_prepack": (_ST, [_P, _P, ctypes.c_float, ctypes.c_int, _I64, _I64, _P, _SZ, _P,
                             ctypes.POINTER(_P)]),
    "vt_fp4_prepack_gate_up": (_ST, [_P, _P, ctypes.c_float, _P, _P, ctypes.c_float, ctypes.c_int,
                                     _I64, _I64, _P, _SZ, _P, ctypes.POINTER(_P)]),
    "vt_fp4_prepack_gate_up_paired": (_ST, [_P, _P, ctypes.c_float, _P, _P, ctypes.c_float,
                                            ctypes.c_int, _I64, _I64, _P, _SZ, _P,
                                            ctypes.POINTER(_P)]),
    "vt_fp4_w4a16_gemm_silu_mul": (_ST, [_P, _I64, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "vt_fp4_prepack_grouped_bytes": (_ST, [ctypes.c_int, _I64, _I64, _I64, ctypes.POINTER(_SZ)]),
    "vt_fp4_prepack_grouped": (_ST, [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P, _SZ, _P,
                                     ctypes.POINTER(_P)]),
    "vt_fp4_moe_workspace_bytes": (_ST, [_P, _I64, _I64, ctypes.POINTER(_SZ)]),
    "vt_fp4_w4a16_gemm_moe": (_ST, [_P, _I64, _I64, _P, _P, _I64, _P, _I64, _P, _SZ, _P]),
    "vt_fp4_destroy": (_ST, [_P]),
    "vt_fp4_shape": (_ST, [_P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(_I64),
                           ctypes.POINTER(_I64)]),
    "vt_fp4_workspace_bytes": (_ST, [_P, _I64, ctypes.POINTER(_SZ)]),
    "vt_fp4_w4a16_gemm": (_ST, [_P, _I64, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "vt_fp4_w4a16_gemm_ex": (_ST, [_P, _I64, _I64, _P, _P, _I64, _P, _SZ, _P,
                                   ctypes.POINTER(GemmOpts)]),
    "vt_fp4_w4a16_gemm_noalloc": (_ST, [_P, _I64, _I64, _P, _P, _I64, _P]),
    "vt_fp4_noalloc_status": (_ST, [_P, ctypes.POINTER(ctypes.c_int)]),
    "vt_fp4_noalloc_test_hooks": (_ST, [ctypes.c_int, ctypes.c_int]),
    "vt_fp4_w4a16_gemm_greedy": (_ST, [_P, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "vt_fp4_workspace_status": (_ST, [_P, _P, ctypes.POINTER(ctypes.c_int)]),
    "vt_fp4_stats": (_ST, [_P, ctypes.POINTER(LaunchInfo)]),
    "vt_fp4_dequant": (_ST, [_P, _P, _P]),
    "vt_fp4_unpack": (_ST, [_P, _P, _P, _P]),
    "vt_fp4_quantize": (_ST, [_P, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P]),
    "vt_fp4_quantize_act": (_ST, [_P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_float, _P, _P,
                                  _P]),
    "vt_fp4_w4a4_gemm": (_ST, [_P, _I64, _I64, _P, ctypes.c_float, _P, _I64, _P, _SZ, _P]),
    "vt_fp4_w4a4_gemm_ex": (_ST, [_P, _I64, _I64, _P, ctypes.c_float, _P, _I64, _P, _SZ, _P,
                                  ctypes.POINTER(GemmOpts)]),
    "vt_fp4_last_error": (ctypes.c_char_p, []),
}

_lib = None


class VtError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Loads libvtfp4.so; raises if it has not been built (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "fp4_weight_only_nvfp4_gb300.build.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != VT_OK:
        msg = lib().vt_fp4_last_error().decode(errors="replace")
        raise VtError(status, where, msg)
