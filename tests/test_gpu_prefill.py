"""GPU: the prefill tile GEMM (tcgen05 tensor cores, M > 16) against the oracle, element by
element, at sizes that span several 128-token and 256-row tiles with ragged tails in M, N and
K; the path forced on small M; fused gate_up against split; run-to-run and grid-independent
bits; activation rows of extreme range; strided operands."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, bf16_host_bits, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu

# (N, K): one row tile; several 256-row tiles with a lone 128-row tile at the end (RT odd);
# a ragged last k tile (K % 64 != 0); rows not a multiple of 128
SHAPES = [(128, 64), (640, 1024), (600, 992), (1000, 2048)]


def _packed(fmt, N, K, tid):
    codes, scales, G = make_weight(fmt, tid, N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    return W, codes, scales, G


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_prefill_matches_oracle(fmt, N, K):
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(70, fmt, 1, N * 7 + K))
    Ms = (17, 128, 300)
    ws = W.new_workspace(max(Ms))
    for M in Ms:
        Ab = make_acts(synth.tensor_id(70, fmt, 2, M * 1000 + N), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W, workspace=ws)
        torch.cuda.synchronize()
        st = W.stats()
        assert st["path"] == 2 and st["m_tile"] == 128
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"prefill fmt={fmt} M={M} N={N} K={K}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_prefill_forced_on_small_m(fmt):
    N, K = 384, 512
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(71, fmt, 1))
    for M in (1, 5, 16):
        Ab = make_acts(synth.tensor_id(71, fmt, 2, M), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W, opts={"force_path": 2})
        torch.cuda.synchronize()
        assert W.stats()["path"] == 2
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"forced prefill M={M}")


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_prefill_fused_gate_up_equals_split(fmt):
    I, K, M = 640, 1024, 200
    gc, gs, gG = make_weight(fmt, synth.tensor_id(72, fmt, synth.ROLE_GATE), I, K)
    uc, us, uG = make_weight(fmt, synth.tensor_id(72, fmt, synth.ROLE_UP), I, K)
    Wf = vt.PackedWeight.gate_up((to_dev(gc), to_dev(gs), gG), (to_dev(uc), to_dev(us), uG), fmt, I, K)
    Wg = vt.PackedWeight.from_codes(to_dev(gc), to_dev(gs), gG, fmt, I, K)
    Wu = vt.PackedWeight.from_codes(to_dev(uc), to_dev(us), uG, fmt, I, K)
    Ab = make_acts(synth.tensor_id(72, fmt, synth.ROLE_A), M, K)
    A = bf16_dev(Ab)
    yf = vt.w4a16_gemm(A, Wf)
    split = torch.cat([vt.w4a16_gemm(A, Wg), vt.w4a16_gemm(A, Wu)], dim=1)
    torch.cuda.synchronize()
    rg, _ = oracle.gemm(fmt, Ab, gc, gs, gG, I)
    ru, _ = oracle.gemm(fmt, Ab, uc, us, uG, I)
    ref = np.concatenate([rg, ru], axis=1)
    check_rows(yf.float().cpu().numpy(), ref, what="fused")
    check_rows(split.float().cpu().numpy(), ref, what="split")
    same = (bf16_host_bits(yf) == bf16_host_bits(split)).mean()
    assert same >= 0.99, same


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_prefill_deterministic_and_grid_independent(fmt):
    """Each output tile is summed by one CTA in a fixed k order, so the bits do not depend
    on the number of CTAs.  Repeated: a CTA that runs many tiles reuses every ring stage
    many times, so a hand-off race between the kernel's roles shows up as changed bits
    (one such race, in the release of the packed-weight stages, changed about a quarter of
    the MXFP4 runs with few CTAs)."""
    N, K, M = 1280, 1536, 260
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(73, fmt, 1))
    Ab = make_acts(synth.tensor_id(73, fmt, 2), M, K)
    A = bf16_dev(Ab)
    ws = W.new_workspace(M)
    first = bf16_host_bits(vt.w4a16_gemm(A, W, workspace=ws))
    for rep in range(8):
        for opts in (None, {"grid": 1}, {"grid": 2}, {"grid": 7}, {"grid": 1000}):
            again = bf16_host_bits(vt.w4a16_gemm(A, W, workspace=ws, opts=opts))
            assert np.array_equal(first, again), (rep, opts)
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    check_rows((first.astype(np.uint32) << 16).view(np.float32), ref, what="deterministic")
    assert vt.workspace_status(ws) == 0


def test_prefill_activation_range_extremes():
    fmt, N, K = vt.NVFP4, 384, 640
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(74, 0, 1))
    base = synth.bf16_bits_to_f32(make_acts(synth.tensor_id(74, 0, 2), 40, K)).astype(np.float64)
    base[0] = 0.0
    base[1] *= 1e-30
    base[2] *= 1e30
    base[3] *= 3e4
    base[4][: K // 2] *= 1e20
    base[5] *= 1e-3
    Ab = torch.tensor(base).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = vt.w4a16_gemm(bf16_dev(Ab), W)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    got = y.float().cpu().numpy()
    assert np.all(got[0] == 0.0)
    check_rows(got, ref, what="extremes")


def test_prefill_strided_operands_and_scalar_stores():
    """lda > K; C with ldc not a multiple of 8 (the epilogue's scalar store path) and
    nothing written past N."""
    fmt, N, K, M = vt.MXFP4, 330, 512, 150
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(75, 0, 1))
    Ab = make_acts(synth.tensor_id(75, 0, 2), M, K)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :K] = bf16_dev(Ab)
    C = torch.full((M, N + 6), 7.0, dtype=torch.bfloat16, device="cuda")  # ldc = 336: vector path
    C2 = torch.full((M, N + 2), 7.0, dtype=torch.bfloat16, device="cuda")  # ldc = 332: scalar path
    vt.w4a16_gemm(big[:, :K], W, out=C[:, :N])
    vt.w4a16_gemm(big[:, :K], W, out=C2[:, :N])
    torch.cuda.synchronize()
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    check_rows(C[:, :N].float().cpu().numpy(), ref, what="strided vec")
    check_rows(C2[:, :N].float().cpu().numpy(), ref, what="strided scalar")
    assert torch.all(C[:, N:] == 7.0) and torch.all(C2[:, N:] == 7.0)
    assert np.array_equal(bf16_host_bits(C[:, :N]), bf16_host_bits(C2[:, :N]))
