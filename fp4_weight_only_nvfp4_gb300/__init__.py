"""GB300-native FP4 weight-only (W4A16) linear layers: NVFP4 and MXFP4 weights against bf16
activations, for LLM decode (M <= 16) and prefill.

This module is a thin binding over the C ABI of ``libvtfp4.so`` (``include/vt_fp4.h``):
PyTorch supplies device memory and streams, every step of the computation runs in the
library's CUDA kernels.  If the library is missing the calls raise; nothing falls back to
PyTorch or the CPU.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import GemmOpts, LaunchInfo, VtError, check, lib

NVFP4, MXFP4 = 0, 1
GROUP = {NVFP4: 16, MXFP4: 32}

__all__ = ["NVFP4", "MXFP4", "GROUP", "PackedWeight", "w4a16_gemm", "w4a16_gemm_noalloc",
           "w4a16_gemm_greedy", "w4a16_gemm_silu_mul", "w4a16_gemm_moe", "w4a4_gemm",
           "quantize_act", "quantize", "prepack_bytes", "workspace_status", "noalloc_status", "VtError",
           "algorithmic_bytes"]


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def algorithmic_bytes(fmt: int, N: int, K: int, M: int) -> int:
    """Bytes a W4A16 call must move at minimum: packed codes N*K/2, one scale byte per group,
    the 4-byte NVFP4 global and the bf16 activations 2*M*K (output bytes not included)."""
    return N * K // 2 + N * K // GROUP[fmt] + (4 if fmt == NVFP4 else 0) + 2 * M * K


def prepack_bytes(fmt: int, N: int, K: int) -> int:
    out = ctypes.c_size_t(0)
    check(lib().vt_fp4_prepack_bytes(fmt, N, K, ctypes.byref(out)), "vt_fp4_prepack_bytes")
    return out.value


class PackedWeight:
    """A weight prepacked into the kernels' tile layout.  Owns its packed device buffer (a
    torch uint8 tensor) and the library handle."""

    def __init__(self, handle: ctypes.c_void_p, packed: torch.Tensor, fmt: int, N: int, K: int):
        self._h = handle
        self.packed = packed
        self.fmt, self.N, self.K = fmt, N, K

    @classmethod
    def from_codes(cls, codes: torch.Tensor, scales: torch.Tensor, global_scale: float, fmt: int,
                   N: int, K: int, stream=None) -> "PackedWeight":
        """codes u8 [N, K/2] (low nibble = even k), scales u8 [N, K/g], both on the GPU."""
        _check_src(codes, scales, N, K, fmt)
        nbytes = prepack_bytes(fmt, N, K)
        packed = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
        h = ctypes.c_void_p(0)
        check(lib().vt_fp4_prepack(_ptr(codes), _ptr(scales), float(global_scale), fmt, N, K,
                                   _ptr(packed), nbytes, _stream(stream), ctypes.byref(h)),
              "vt_fp4_prepack")
        return cls(h, packed, fmt, N, K)

    @classmethod
    def gate_up(cls, gate: tuple, up: tuple, fmt: int, I: int, K: int, stream=None,
                paired: bool = False) -> "PackedWeight":
        """Fused gate_up: ``gate``/``up`` are (codes, scales, global); N = 2*I.  ``paired``
        packs gate and up rows side by side for the SiLU-and-multiply epilogue
        (vt_fp4_prepack_gate_up_paired)."""
        (gc, gs, gg), (uc, us, ug) = gate, up
        _check_src(gc, gs, I, K, fmt)
        _check_src(uc, us, I, K, fmt)
        nbytes = prepack_bytes(fmt, 2 * I, K)
        packed = torch.empty(nbytes, dtype=torch.uint8, device=gc.device)
        h = ctypes.c_void_p(0)
        name = "vt_fp4_prepack_gate_up_paired" if paired else "vt_fp4_prepack_gate_up"
        check(getattr(lib(), name)(_ptr(gc), _ptr(gs), float(gg), _ptr(uc), _ptr(us),
                                   float(ug), fmt, I, K, _ptr(packed), nbytes,
                                   _stream(stream), ctypes.byref(h)), name)
        W = cls(h, packed, fmt, 2 * I, K)
        W.I = I
        W.paired = paired
        return W

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("PackedWeight has been closed")
        return self._h

    def workspace_bytes(self, M_max: int) -> int:
        out = ctypes.c_size_t(0)
        check(lib().vt_fp4_workspace_bytes(self.handle, M_max, ctypes.byref(out)),
              "vt_fp4_workspace_bytes")
        return out.value

    def new_workspace(self, M_max: int) -> torch.Tensor:
        """A zeroed workspace for calls with M <= M_max (zero once; the library keeps its
        counters usable from call to call, for this or any other weight it is large enough for)."""
        return torch.zeros(self.workspace_bytes(M_max), dtype=torch.uint8,
                           device=self.packed.device)

    @classmethod
    def grouped(cls, codes: torch.Tensor, scales: torch.Tensor, globals_: list, fmt: int,
                E: int, N: int, K: int, stream=None) -> "PackedWeight":
        """E experts of N x K: codes [E, N, K/2], scales [E, N, K/g], one global per expert
        (vt_fp4_prepack_grouped)."""
        if codes.shape != (E, N, K // 2) or scales.shape != (E, N, K // GROUP[fmt]):
            raise ValueError("codes [E, N, K/2] and scales [E, N, K/g] expected")
        _check_src(codes, scales, E * N, K, fmt)
        if len(globals_) != E:
            raise ValueError("one global per expert expected")
        out = ctypes.c_size_t(0)
        check(lib().vt_fp4_prepack_grouped_bytes(fmt, E, N, K, ctypes.byref(out)),
              "vt_fp4_prepack_grouped_bytes")
        packed = torch.empty(out.value, dtype=torch.uint8, device=codes.device)
        g = (ctypes.c_float * E)(*[float(x) for x in globals_])
        h = ctypes.c_void_p(0)
        check(lib().vt_fp4_prepack_grouped(_ptr(codes.contiguous()), _ptr(scales.contiguous()),
                                           ctypes.cast(g, ctypes.c_void_p), fmt, E, N, K,
                                           _ptr(packed), out.value, _stream(stream),
                                           ctypes.byref(h)), "vt_fp4_prepack_grouped")
        W = cls(h, packed, fmt, N, K)
        W.E = E
        return W

    def moe_workspace(self, M_max: int, topk: int) -> torch.Tensor:
        out = ctypes.c_size_t(0)
        check(lib().vt_fp4_moe_workspace_bytes(self.handle, M_max, topk, ctypes.byref(out)),
              "vt_fp4_moe_workspace_bytes")
        return torch.zeros(out.value, dtype=torch.uint8, device=self.packed.device)

    def dequant(self, stream=None) -> torch.Tensor:
        out = torch.empty((getattr(self, "E", 1) * self.N, self.K), dtype=torch.float32,
                          device=self.packed.device)
        check(lib().vt_fp4_dequant(self.handle, _ptr(out), _stream(stream)), "vt_fp4_dequant")
        return out

    def unpack(self, stream=None):
        dev = self.packed.device
        rows = getattr(self, "E", 1) * self.N
        codes = torch.empty((rows, self.K // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((rows, self.K // GROUP[self.fmt]), dtype=torch.uint8, device=dev)
        check(lib().vt_fp4_unpack(self.handle, _ptr(codes), _ptr(scales), _stream(stream)),
              "vt_fp4_unpack")
        return codes, scales

    def stats(self) -> dict:
        info = LaunchInfo()
        check(lib().vt_fp4_stats(self.handle, ctypes.byref(info)), "vt_fp4_stats")
        return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}

    def close(self) -> None:
        if self._h:
            lib().vt_fp4_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check_src(codes, scales, N, K, fmt):
    if codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
        raise TypeError("codes and scales must be uint8 tensors")
    if not (codes.is_cuda and scales.is_cuda and codes.is_contiguous() and scales.is_contiguous()):
        raise ValueError("codes and scales must be contiguous CUDA tensors")
    if codes.numel() != N * K // 2 or scales.numel() != N * K // GROUP[fmt]:
        raise ValueError("codes/scales sizes do not match N and K")


def _check_A(A: torch.Tensor, W: "PackedWeight"):
    if A.dtype != torch.bfloat16 or A.dim() != 2 or A.shape[1] != W.K or A.stride(1) != 1:
        raise ValueError("A must be a bf16 [M, K] tensor with unit inner stride")


def _check_out(out: torch.Tensor, rows: int, cols: int, name: str = "out"):
    """The kernels write rows x cols bf16 values at the given row stride: a smaller or
    differently typed tensor would be written past its end."""
    if out.dtype != torch.bfloat16 or out.dim() != 2 or tuple(out.shape) != (rows, cols) \
            or out.stride(1) != 1:
        raise ValueError(f"{name} must be a bf16 [{rows}, {cols}] tensor with unit inner stride")


def _check_device(W: "PackedWeight", **tensors):
    """Every tensor handed to the kernels must live on the weight's GPU: a host tensor or
    another device's memory would reach the kernels as a wild address."""
    dev = W.packed.device
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be a CUDA tensor on {dev} (got {t.device})")
        if name == "workspace" and (t.dtype != torch.uint8 or not t.is_contiguous()):
            raise ValueError("workspace must be a contiguous uint8 tensor")


def _opts(opts: dict | None):
    if not opts:
        return None
    return GemmOpts(int(opts.get("grid", 0)), int(opts.get("warps", 0)),
                    int(opts.get("stages", 0)), int(opts.get("force_path", 0)),
                    int(opts.get("wait_limit_us", 0)), int(opts.get("withhold_weights", 0)))


def w4a16_gemm(A: torch.Tensor, W: PackedWeight, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, stream=None,
               opts: dict | None = None) -> torch.Tensor:
    """out[M, N] (bf16) = A[M, K] (bf16) . W^T, fp32 accumulation, on the library's kernels."""
    _check_A(A, W)
    _check_device(W, A=A, out=out, workspace=workspace)
    M = A.shape[0]
    if out is None:
        out = torch.empty((M, W.N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, W.N)
    if workspace is None:
        workspace = W.new_workspace(M)
    o = _opts(opts)
    check(lib().vt_fp4_w4a16_gemm_ex(_ptr(A), M, A.stride(0), W.handle, _ptr(out),
                                     out.stride(0), _ptr(workspace), workspace.numel(),
                                     _stream(stream), ctypes.byref(o) if o else None),
          "vt_fp4_w4a16_gemm")
    return out


def w4a4_gemm(A: torch.Tensor, W: PackedWeight, input_scale: float = 1.0,
              out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              stream=None, opts: dict | None = None) -> torch.Tensor:
    """The W4A4 arm: out[M, N] (bf16) = Q(A) . W^T with the activations quantised to W's
    block format (NVFP4 with the activation global ``input_scale``; MXFP4: 1.0)."""
    _check_A(A, W)
    _check_device(W, A=A, out=out, workspace=workspace)
    M = A.shape[0]
    if out is None:
        out = torch.empty((M, W.N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, W.N)
    if workspace is None:
        workspace = W.new_workspace(M)
    o = _opts(opts)
    check(lib().vt_fp4_w4a4_gemm_ex(_ptr(A), M, A.stride(0), W.handle, float(input_scale),
                                    _ptr(out), out.stride(0), _ptr(workspace),
                                    workspace.numel(), _stream(stream),
                                    ctypes.byref(o) if o else None), "vt_fp4_w4a4_gemm")
    return out


def quantize_act(A: torch.Tensor, fmt: int, input_scale: float = 1.0, stream=None):
    """The W4A4 activation quantiser: A bf16 [M, K] (CUDA, unit inner stride) ->
    (codes u8 [M, K/2], scales u8 [M, K/g])."""
    if A.dtype != torch.bfloat16 or A.dim() != 2 or A.stride(1) != 1 or not A.is_cuda:
        raise ValueError("A must be a bf16 CUDA [M, K] tensor with unit inner stride")
    M, K = A.shape
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=A.device)
    scales = torch.empty((M, K // GROUP[fmt]), dtype=torch.uint8, device=A.device)
    check(lib().vt_fp4_quantize_act(_ptr(A), M, A.stride(0), K, fmt, float(input_scale),
                                    _ptr(codes), _ptr(scales), _stream(stream)),
          "vt_fp4_quantize_act")
    return codes, scales


def w4a16_gemm_moe(A: torch.Tensor, W: PackedWeight, topk_ids: torch.Tensor,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Mixture-of-experts decode GEMM: out[m * topk + j] = A[m] . W_e^T with
    e = topk_ids[m, j] (see vt_fp4_w4a16_gemm_moe in include/vt_fp4.h)."""
    _check_A(A, W)
    if topk_ids.dtype != torch.int32 or topk_ids.dim() != 2 or topk_ids.shape[0] != A.shape[0]:
        raise ValueError("topk_ids must be an int32 [M, topk] tensor")
    _check_device(W, A=A, topk_ids=topk_ids, out=out, workspace=workspace)
    M, topk = topk_ids.shape
    topk_ids = topk_ids.contiguous()
    if out is None:
        out = torch.empty((M * topk, W.N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M * topk, W.N)
    if workspace is None:
        workspace = W.moe_workspace(max(M, 1), topk)
    check(lib().vt_fp4_w4a16_gemm_moe(_ptr(A), M, A.stride(0), W.handle, _ptr(topk_ids), topk,
                                      _ptr(out), out.stride(0), _ptr(workspace),
                                      workspace.numel(), _stream(stream)),
          "vt_fp4_w4a16_gemm_moe")
    return out


def w4a16_gemm_silu_mul(A: torch.Tensor, W: PackedWeight, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[M, I] (bf16) = silu(gate) * up of a paired gate_up weight, in one call (see
    vt_fp4_w4a16_gemm_silu_mul in include/vt_fp4.h)."""
    _check_A(A, W)
    _check_device(W, A=A, out=out, workspace=workspace)
    M = A.shape[0]
    if out is None:
        out = torch.empty((M, W.N // 2), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, W.N // 2)
    if workspace is None:
        workspace = W.new_workspace(M)
    check(lib().vt_fp4_w4a16_gemm_silu_mul(_ptr(A), M, A.stride(0), W.handle, _ptr(out),
                                           out.stride(0), _ptr(workspace), workspace.numel(),
                                           _stream(stream)), "vt_fp4_w4a16_gemm_silu_mul")
    return out


def w4a16_gemm_greedy(A: torch.Tensor, W: PackedWeight, workspace: torch.Tensor | None = None,
                      stream=None, want_value: bool = True, token: torch.Tensor | None = None):
    """Greedy head (M <= 16): per token, the index (int32 [M]) of the largest bf16 output of
    A . W^T, ties to the lowest index, and that value (fp32 [M]) -- without writing the
    outputs.  ``token``: an optional int32 [M] output tensor.  See vt_fp4_w4a16_gemm_greedy
    in include/vt_fp4.h."""
    _check_A(A, W)
    _check_device(W, A=A, token=token, workspace=workspace)
    M = A.shape[0]
    if token is None:
        token = torch.empty(M, dtype=torch.int32, device=A.device)
    elif token.dtype != torch.int32 or token.shape != (M,) or not token.is_contiguous():
        raise ValueError("token must be a contiguous int32 [M] tensor")
    value = torch.empty(M, dtype=torch.float32, device=A.device) if want_value else None
    if workspace is None:
        workspace = W.new_workspace(M)
    check(lib().vt_fp4_w4a16_gemm_greedy(_ptr(A), M, A.stride(0), W.handle, _ptr(token),
                                         _ptr(value), _ptr(workspace), workspace.numel(),
                                         _stream(stream)), "vt_fp4_w4a16_gemm_greedy")
    return token, value


def w4a16_gemm_noalloc(A: torch.Tensor, W: PackedWeight, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """The decode GEMM (M <= 16) on the library's fixed scratch area instead of a caller
    workspace, for callers that cannot allocate device memory (see vt_fp4_w4a16_gemm_noalloc
    in include/vt_fp4.h).  Calls must not overlap on the GPU."""
    _check_A(A, W)
    _check_device(W, A=A, out=out)
    M = A.shape[0]
    if out is None:
        out = torch.empty((M, W.N), dtype=torch.bfloat16, device=A.device)
    _check_out(out, M, W.N)
    check(lib().vt_fp4_w4a16_gemm_noalloc(_ptr(A), M, A.stride(0), W.handle, _ptr(out),
                                          out.stride(0), _stream(stream)),
          "vt_fp4_w4a16_gemm_noalloc")
    return out


def noalloc_status(stream=None) -> int:
    """The no-alloc scratch area's status word on the current device (0, or VT_ERR_TIMEOUT
    when a bounded wait of an earlier w4a16_gemm_noalloc call gave up); read and cleared,
    synchronising the stream."""
    st = ctypes.c_int(0)
    check(lib().vt_fp4_noalloc_status(_stream(stream), ctypes.byref(st)), "vt_fp4_noalloc_status")
    return st.value


def workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """The workspace's status word (0, or the code a kernel recorded there); synchronises
    the stream."""
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    st = ctypes.c_int(0)
    check(lib().vt_fp4_workspace_status(_ptr(workspace), _stream(stream), ctypes.byref(st)),
          "vt_fp4_workspace_status")
    return st.value


def quantize(W: torch.Tensor, fmt: int, stream=None):
    """Quantise a bf16 [N, K] CUDA tensor: returns (codes u8 [N, K/2], scales u8 [N, K/g],
    global fp32 tensor [1] (1.0 for MXFP4))."""
    if W.dtype != torch.bfloat16 or W.dim() != 2 or not W.is_contiguous() or not W.is_cuda:
        raise ValueError("W must be a contiguous bf16 CUDA [N, K] tensor")
    N, K = W.shape
    dev = W.device
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // GROUP[fmt]), dtype=torch.uint8, device=dev)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    scratch = torch.empty(16, dtype=torch.uint8, device=dev)
    check(lib().vt_fp4_quantize(_ptr(W), N, K, fmt, _ptr(codes), _ptr(scales), _ptr(g),
                                _ptr(scratch), _stream(stream)), "vt_fp4_quantize")
    return codes, scales, g
