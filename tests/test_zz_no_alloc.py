"""GPU: the decode GEMM entry point for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: their device memory belongs to another
allocator (a serving engine that reserves its HBM up front, a plugin whose host forbids
foreign allocations) or their call path must not depend on a runtime allocation.  For them
vt_fp4_w4a16_gemm_noalloc runs the decode GEMM on a fixed scratch area inside the library
instead of a caller workspace.  These tests call it through the C ABI: twice in a row with
different weights and batch sizes against the regular entry point (vt_fp4_w4a16_gemm with a
caller workspace), against the oracle at every token count it serves (activations converted
inside the decode kernel at small M * K, by the pre-pass otherwise; 8- and 16-token tiles),
its rejections, and a bounded wait that runs out (reported by vt_fp4_noalloc_status, after
which the next call is correct again).  The file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import TOL, bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(A: torch.Tensor, W, out: torch.Tensor) -> int:
    s = torch.cuda.current_stream().cuda_stream
    return _lib.lib().vt_fp4_w4a16_gemm_noalloc(
        ctypes.c_void_p(A.data_ptr()), A.shape[0], A.stride(0), W.handle,
        ctypes.c_void_p(out.data_ptr()), out.stride(0), ctypes.c_void_p(s))


def _status() -> int:
    st = ctypes.c_int(-1)
    s = torch.cuda.current_stream().cuda_stream
    assert _lib.lib().vt_fp4_noalloc_status(ctypes.c_void_p(s), ctypes.byref(st)) == _lib.VT_OK
    return st.value


def _close(got: torch.Tensor, ref: torch.Tensor) -> None:
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    for m in range(r.shape[0]):
        den = np.abs(r[m]).max()
        err = np.abs(g[m] - r[m]).max()
        assert err <= TOL * den, (m, err, den)


def _weight(fmt, N, K, i):
    codes, scales, G = make_weight(fmt, synth.tensor_id(90, i, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    return W, codes, scales, G


def test_noalloc_matches_workspace_gemm_twice_in_a_row():
    cases = [(vt.NVFP4, 1000, 2048, 5), (vt.MXFP4, 3072, 4096, 8)]
    built = []
    for i, (fmt, N, K, M) in enumerate(cases):
        W, _, _, _ = _weight(fmt, N, K, i)
        A = bf16_dev(make_acts(synth.tensor_id(90, i, 2), M, K))
        built.append((W, A))
    for W, A in built:  # two calls in a row, the second reusing the scratch of the first
        out = torch.full((A.shape[0], W.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(A, W, out) == _lib.VT_OK, _lib.lib().vt_fp4_last_error()
        ref = vt.w4a16_gemm(A, W)
        torch.cuda.synchronize()
        _close(out, ref)
    assert _status() == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_noalloc_matches_oracle_every_mode(fmt):
    N, K = 1000, 2048  # M = 1, 2: converted inside the kernel; 5: pre-pass; 13, 16: 16-token tile
    W, codes, scales, G = _weight(fmt, N, K, 10 + fmt)
    for M in (1, 2, 5, 13, 16):
        Ab = make_acts(synth.tensor_id(90, 10 + fmt, 3, M), M, K)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(bf16_dev(Ab), W, out) == _lib.VT_OK, _lib.lib().vt_fp4_last_error()
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(out.float().cpu().numpy(), ref, what=f"noalloc fmt={fmt} M={M}")
        st = W.stats()
        assert st["path"] == 1 and st["m_tile"] == (8 if M <= 8 else 16)
        assert st["launches"] == (1 if M <= 2 else 2)  # resident mode: no pre-pass kernel
    assert _status() == 0


def _raw_weight(fmt, N, K, seed):
    """Random codes and mid-range scales: enough for the argument checks."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(0x30, 0x40, size=(N, K // vt.GROUP[fmt]), dtype=np.uint8)
    return vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, fmt, N, K)


def test_noalloc_rejects_what_the_scratch_cannot_hold():
    # 16 tokens of K = 98304: converted activations 3 MiB plus split-K partials 1.5 MiB > 4 MiB
    W = _raw_weight(vt.NVFP4, 128, 98304, 1)
    A = bf16_dev(make_acts(synth.tensor_id(90, 9, 2), 16, 98304))
    out = torch.empty((16, 128), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, W, out) == _lib.VT_ERR_UNSUPPORTED
    assert b"scratch" in _lib.lib().vt_fp4_last_error()
    # one token of K = 131072 would fit the scratch, but K > 110000 is refused as elsewhere
    Wk = _raw_weight(vt.NVFP4, 128, 131072, 2)
    A1 = bf16_dev(make_acts(synth.tensor_id(90, 9, 3), 1, 131072))
    out1 = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A1, Wk, out1) == _lib.VT_ERR_UNSUPPORTED
    assert b"110000" in _lib.lib().vt_fp4_last_error()
    # more than 16 tokens is the tile path's range, which needs a workspace
    W2 = _raw_weight(vt.NVFP4, 64, 4096, 3)
    A17 = bf16_dev(make_acts(synth.tensor_id(90, 9, 4), 17, 4096))
    out17 = torch.empty((17, 64), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A17, W2, out17) == _lib.VT_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_noalloc_rejects_a_grouped_weight():
    E, N, K = 2, 128, 256
    cs, ss = [], []
    for e in range(E):
        c, s, _ = make_weight(vt.MXFP4, synth.tensor_id(90, 20, e), N, K)
        cs.append(c)
        ss.append(s)
    W = vt.PackedWeight.grouped(to_dev(np.stack(cs)), to_dev(np.stack(ss)), [1.0] * E, vt.MXFP4,
                                E, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(90, 20, 9), 2, K))
    out = torch.empty((2, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(A, W, out) == _lib.VT_ERR_INVALID_ARG
    assert b"grouped" in _lib.lib().vt_fp4_last_error()


def test_noalloc_wait_that_runs_out_is_reported_then_recovers():
    N, K = 1000, 2048
    W, codes, scales, G = _weight(vt.NVFP4, N, K, 30)
    lib = _lib.lib()
    try:
        for M in (1, 12):  # resident mode and the pre-pass path
            Ab = make_acts(synth.tensor_id(90, 30, 4, M), M, K)
            A = bf16_dev(Ab)
            out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            assert lib.vt_fp4_noalloc_test_hooks(20000, 1) == _lib.VT_OK  # 20 ms, no copies
            assert _noalloc(A, W, out) == _lib.VT_OK
            torch.cuda.synchronize()
            assert _status() == _lib.VT_ERR_TIMEOUT
            assert _status() == 0  # read once, then cleared
            assert lib.vt_fp4_noalloc_test_hooks(0, 0) == _lib.VT_OK
            assert _noalloc(A, W, out) == _lib.VT_OK
            torch.cuda.synchronize()
            ref, _ = oracle.gemm(vt.NVFP4, Ab, codes, scales, G, N)
            check_rows(out.float().cpu().numpy(), ref, what=f"after timeout M={M}")
            assert _status() == 0
    finally:
        lib.vt_fp4_noalloc_test_hooks(0, 0)
