"""GPU: the decode GEMM entry point for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: their device memory belongs to another
allocator (a serving engine that reserves its HBM up front, a plugin whose host forbids
foreign allocations) or their call path must not depend on a runtime allocation.  For them
vt_fp4_w4a16_gemm_noalloc runs the decode GEMM on a fixed scratch area inside the library
instead of a caller workspace.  This test calls it through the C ABI, twice in a row with
different weights and batch sizes, and checks each output against the regular entry point
(vt_fp4_w4a16_gemm with a caller workspace) on the same inputs, with the same tolerance the
parity tests use.  It lives in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import TOL, bf16_dev, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(A: torch.Tensor, W, out: torch.Tensor) -> int:
    s = torch.cuda.current_stream().cuda_stream
    return _lib.lib().vt_fp4_w4a16_gemm_noalloc(
        ctypes.c_void_p(A.data_ptr()), A.shape[0], A.stride(0), W.handle,
        ctypes.c_void_p(out.data_ptr()), out.stride(0), ctypes.c_void_p(s))


def _close(got: torch.Tensor, ref: torch.Tensor) -> None:
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    for m in range(r.shape[0]):
        den = np.abs(r[m]).max()
        err = np.abs(g[m] - r[m]).max()
        assert err <= TOL * den, (m, err, den)


def test_noalloc_matches_workspace_gemm_twice_in_a_row():
    cases = [(vt.NVFP4, 1000, 2048, 5), (vt.MXFP4, 3072, 4096, 8)]
    built = []
    for i, (fmt, N, K, M) in enumerate(cases):
        codes, scales, G = make_weight(fmt, synth.tensor_id(90, i, 1), N, K)
        W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
        A = bf16_dev(make_acts(synth.tensor_id(90, i, 2), M, K))
        built.append((W, A))
    for W, A in built:  # two calls in a row, the second reusing the scratch of the first
        out = torch.full((A.shape[0], W.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(A, W, out) == _lib.VT_OK, _lib.lib().vt_fp4_last_error()
        ref = vt.w4a16_gemm(A, W)
        torch.cuda.synchronize()
        _close(out, ref)


def test_noalloc_rejects_what_the_scratch_cannot_hold():
    N, K = 128, 131072  # the converted activations alone need 16 x 131072 x 2 B = 4 MiB
    codes, scales, G = make_weight(vt.NVFP4, synth.tensor_id(90, 9, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, vt.NVFP4, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(90, 9, 2), 16, K))
    out = torch.empty((16, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, W, out) == _lib.VT_ERR_UNSUPPORTED
    assert b"scratch" in _lib.lib().vt_fp4_last_error()
    A17 = bf16_dev(make_acts(synth.tensor_id(90, 9, 3), 17, K))
    out17 = torch.empty((17, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A17, W, out17) == _lib.VT_ERR_UNSUPPORTED
