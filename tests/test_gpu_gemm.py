"""GPU: the decode GEMM against the oracle, element by element, at sizes the oracle finishes in
seconds that span several tiles and ragged tails; fused gate_up against split; determinism,
launch-shape independence within tolerance, workspace reuse and edge cases."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, bf16_host_bits, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(300, 160), (2048, 1024), (1000, 4096), (130, 64), (384, 17408 // 4)]


def _packed(fmt, N, K, tid):
    codes, scales, G = make_weight(fmt, tid, N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    return W, codes, scales, G


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_decode_gemm_matches_oracle(fmt, N, K):
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(60, fmt, 1, N * 7 + K))
    ws = W.new_workspace(16)
    for M in (1, 2, 3, 5, 8, 9, 13, 16):
        Ab = make_acts(synth.tensor_id(60, fmt, 2, M * 1000 + N), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W, workspace=ws)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"fmt={fmt} M={M} N={N} K={K}")
        st = W.stats()
        assert st["path"] == 1 and st["m_tile"] == (8 if M <= 8 else 16)
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_fused_gate_up_equals_split(fmt):
    I, K = 1536, 2048
    gc, gs, gG = make_weight(fmt, synth.tensor_id(61, fmt, synth.ROLE_GATE), I, K)
    uc, us, uG = make_weight(fmt, synth.tensor_id(61, fmt, synth.ROLE_UP), I, K)
    Wf = vt.PackedWeight.gate_up((to_dev(gc), to_dev(gs), gG), (to_dev(uc), to_dev(us), uG), fmt, I, K)
    Wg = vt.PackedWeight.from_codes(to_dev(gc), to_dev(gs), gG, fmt, I, K)
    Wu = vt.PackedWeight.from_codes(to_dev(uc), to_dev(us), uG, fmt, I, K)
    same = total = 0
    for M in (1, 4, 8, 16):
        Ab = make_acts(synth.tensor_id(61, fmt, synth.ROLE_A, M), M, K)
        A = bf16_dev(Ab)
        yf = vt.w4a16_gemm(A, Wf)
        yg = vt.w4a16_gemm(A, Wg)
        yu = vt.w4a16_gemm(A, Wu)
        torch.cuda.synchronize()
        split = torch.cat([yg, yu], dim=1)
        rg, _ = oracle.gemm(fmt, Ab, gc, gs, gG, I)
        ru, _ = oracle.gemm(fmt, Ab, uc, us, uG, I)
        ref = np.concatenate([rg, ru], axis=1)
        check_rows(yf.float().cpu().numpy(), ref, what="fused")
        check_rows(split.float().cpu().numpy(), ref, what="split")
        same += int((bf16_host_bits(yf) == bf16_host_bits(split)).sum())
        total += split.numel()
    # the pages' criterion for fused vs split: >= 99% bit-exact
    assert same / total >= 0.99, same / total


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_deterministic_and_launch_shape_independent(fmt):
    N, K = 1280, 3072
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(62, fmt, 1))
    ws = W.new_workspace(16)
    for M in (1, 6, 16):
        Ab = make_acts(synth.tensor_id(62, fmt, 2, M), M, K)
        A = bf16_dev(Ab)
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        first = bf16_host_bits(vt.w4a16_gemm(A, W, workspace=ws))
        for _ in range(3):
            again = bf16_host_bits(vt.w4a16_gemm(A, W, workspace=ws))
            assert np.array_equal(first, again)  # same launch shape -> same bits
        for opts in ({"grid": 1}, {"grid": 7}, {"grid": 300}, {"warps": 4}, {"stages": 2},
                     {"stages": 3, "warps": 8}, {"grid": 512}, {"warps": 4, "stages": 6}):
            y = vt.w4a16_gemm(A, W, workspace=ws, opts=opts)
            torch.cuda.synchronize()
            check_rows(y.float().cpu().numpy(), ref, what=f"{opts}")
    assert vt.workspace_status(ws) == 0


def test_strided_operands_and_empty_batch():
    fmt, N, K = vt.NVFP4, 520, 640
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(63, 0, 1))
    M = 5
    Ab = make_acts(synth.tensor_id(63, 0, 2), M, K)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :K] = bf16_dev(Ab)
    A = big[:, :K]  # lda = K + 64
    C = torch.full((M, N + 10), 7.0, dtype=torch.bfloat16, device="cuda")
    vt.w4a16_gemm(A, W, out=C[:, :N])
    torch.cuda.synchronize()
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    check_rows(C[:, :N].float().cpu().numpy(), ref, what="strided")
    assert torch.all(C[:, N:] == 7.0)  # nothing written past N
    empty = vt.w4a16_gemm(torch.empty((0, K), dtype=torch.bfloat16, device="cuda"), W)
    assert empty.shape == (0, N)


def test_activation_range_extremes():
    """Rows of zeros, tiny (1e-30) and huge (1e30) activations, and a row whose k tiles differ
    by 1e20: the per-(token, k tile) power-of-two conversion keeps every row within tolerance
    (and zero rows exactly zero)."""
    fmt, N, K = vt.NVFP4, 256, 512
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(64, 0, 1))
    base = synth.bf16_bits_to_f32(make_acts(synth.tensor_id(64, 0, 2), 6, K)).astype(np.float64)
    rows = [np.zeros(K), base[1] * 1e-30, base[2] * 1e30, base[3] * 3e4, base[4], base[5] * 1e-3]
    rows[4][: K // 2] *= 1e20  # two halves of one row 20 orders of magnitude apart
    A = np.stack(rows)
    Ab = torch.tensor(A).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = vt.w4a16_gemm(bf16_dev(Ab), W)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    got = y.float().cpu().numpy()
    assert np.all(got[0] == 0.0)
    check_rows(got, ref, what="extremes")


def test_workspace_reuse_across_shapes():
    fmt = vt.MXFP4
    Ws = [_packed(fmt, N, K, synth.tensor_id(65, i, 1)) for i, (N, K) in
          enumerate([(700, 1024), (4096, 512), (256, 8192)])]
    size = max(W.workspace_bytes(16) for W, *_ in Ws)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for rep in range(3):
        for i, (W, codes, scales, G) in enumerate(Ws):
            M = (rep * 5 + i * 3) % 16 + 1
            Ab = make_acts(synth.tensor_id(65, i, 2, rep), M, W.K)
            y = vt.w4a16_gemm(bf16_dev(Ab), W, workspace=ws)
            torch.cuda.synchronize()
            ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, W.N)
            check_rows(y.float().cpu().numpy(), ref, what=f"reuse {i} {rep}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", [(2048, 1024), (600, 992), (1000, 4096), (384, 12288)])
def test_resident_activations_equal_prepass(fmt, N, K):
    """Small M * K: the decode kernel converts the activations into shared memory itself (one
    launch); forcing the pre-pass (force_path 3, two launches) must give the same bits, and
    both match the oracle.  Rows include zeros and magnitudes far apart."""
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(64, fmt, 1, N + K))
    ws = W.new_workspace(16)
    for M in (1, 2, 3, 4):
        x = synth.bf16_bits_to_f32(make_acts(synth.tensor_id(64, fmt, 2, M * 100 + K), M, K))
        x = x.astype(np.float64)
        if M >= 3:
            x[1] = 0.0
            x[2][: K // 3] *= 1e20
        Ab = torch.tensor(x).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        A = bf16_dev(Ab)
        y_res = vt.w4a16_gemm(A, W, workspace=ws)
        launches_res = W.stats()["launches"]
        y_pre = vt.w4a16_gemm(A, W, workspace=ws, opts={"force_path": 3})
        launches_pre = W.stats()["launches"]
        torch.cuda.synchronize()
        resident = M * ((K + 63) // 64) * 128 <= 16 * 1024
        assert launches_res == (1 if resident else 2) and launches_pre == 2, (M, launches_res)
        assert np.array_equal(bf16_host_bits(y_res), bf16_host_bits(y_pre)), f"M={M}"
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y_res.float().cpu().numpy(), ref, what=f"resident fmt={fmt} M={M} N={N} K={K}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_resident_activations_strided(fmt):
    """The in-kernel activation conversion reads A with its own leading dimension."""
    N, K = 640, 1024
    W, codes, scales, G = _packed(fmt, N, K, synth.tensor_id(65, fmt, 1))
    for M in (1, 2):
        Ab = make_acts(synth.tensor_id(65, fmt, 2, M), M, K)
        big = torch.full((M, K + 72), 3.0, dtype=torch.bfloat16, device="cuda")
        big[:, :K] = bf16_dev(Ab)
        y = vt.w4a16_gemm(big[:, :K], W)
        torch.cuda.synchronize()
        assert W.stats()["launches"] == 1  # resident mode
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"resident strided M={M}")
