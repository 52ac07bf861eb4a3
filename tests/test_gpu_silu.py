"""GPU: the paired gate_up layout and the SiLU-and-multiply epilogue.

The paired prepack is checked bit-exactly through unpack and dequant against the gate and
up sources; vt_fp4_w4a16_gemm_silu_mul against the oracle's silu(g) * u (fp64 from the
oracle's fp32 gate and up sums, one rounding) within the GEMM tolerance, on the decode
(M <= 16) and tile (M > 16) paths; the plain GEMM on a paired handle against the stacked
gate_up handle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import bf16_dev, bf16_host_bits, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _pair(fmt, I, K, tag):
    g = make_weight(fmt, synth.tensor_id(88, tag, synth.ROLE_GATE, I), I, K)
    u = make_weight(fmt, synth.tensor_id(88, tag, synth.ROLE_UP, I), I, K)
    dev = lambda t: (to_dev(t[0]), to_dev(t[1]), t[2])
    Wp = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K, paired=True)
    Ws = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K)
    return g, u, Wp, Ws


def _oracle_silu(fmt, Ab, g, u, I):
    yg, _ = oracle.gemm(fmt, Ab, g[0], g[1], g[2], I)
    yu, _ = oracle.gemm(fmt, Ab, u[0], u[1], u[2], I)
    return oracle.bf16_to_f32(oracle.silu_mul(np.concatenate([yg, yu], axis=1)))


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("I", [64, 100, 300])
def test_paired_prepack_round_trip(fmt, I):
    K = 512
    g, u, Wp, Ws = _pair(fmt, I, K, 1)
    codes, scales = Wp.unpack()
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), np.concatenate([g[0], u[0]]))
    assert np.array_equal(scales.cpu().numpy(), np.concatenate([g[1], u[1]]))
    assert torch.equal(Wp.dequant(), Ws.dequant())


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("I,K", [(100, 512), (640, 1024), (1000, 2048)])
def test_silu_mul_matches_oracle(fmt, I, K):
    g, u, Wp, _ = _pair(fmt, I, K, 2)
    ws = Wp.new_workspace(200)
    for M in (1, 5, 16, 40, 200):
        Ab = make_acts(synth.tensor_id(88, fmt, synth.ROLE_A, M * 10 + I), M, K)
        y = vt.w4a16_gemm_silu_mul(bf16_dev(Ab), Wp, workspace=ws)
        torch.cuda.synchronize()
        assert Wp.stats()["path"] == (1 if M <= 16 else 2)
        check_rows(y.float().cpu().numpy(), _oracle_silu(fmt, Ab, g, u, I),
                   what=f"silu fmt={fmt} I={I} K={K} M={M}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_plain_gemm_on_paired_weight(fmt):
    I, K = 300, 1024
    g, u, Wp, Ws = _pair(fmt, I, K, 3)
    for M in (3, 16, 70):
        Ab = make_acts(synth.tensor_id(88, fmt, 9, M), M, K)
        A = bf16_dev(Ab)
        yp = vt.w4a16_gemm(A, Wp)
        ys = vt.w4a16_gemm(A, Ws)
        torch.cuda.synchronize()
        rg, _ = oracle.gemm(fmt, Ab, g[0], g[1], g[2], I)
        ru, _ = oracle.gemm(fmt, Ab, u[0], u[1], u[2], I)
        ref = np.concatenate([rg, ru], axis=1)
        check_rows(yp.float().cpu().numpy(), ref, what=f"paired plain M={M}")
        same = (bf16_host_bits(yp) == bf16_host_bits(ys)).mean()
        assert same >= 0.99, same


def test_silu_mul_needs_a_paired_weight():
    fmt, I, K = vt.NVFP4, 128, 256
    _, _, _, Ws = _pair(fmt, I, K, 4)
    A = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.VtError) as e:
        vt.w4a16_gemm_silu_mul(A, Ws)
    assert e.value.status == _lib.VT_ERR_INVALID_ARG
