"""GPU: the W4A4 arm against the oracle.  The activation quantiser's codes and scales must
match the oracle's bit for bit (both take the decisions in fp32); the W4A4 GEMM is checked
element by element with the W4A16 tolerance on both paths (decode M <= 16, tensor-core tile
kernel above), across several tiles with ragged M, N and K; inputs with extreme ranges,
zero rows and non-finite values; argument rejection."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu

ALPHAS = {vt.NVFP4: [0.0078125, 0.37, 1e-3], vt.MXFP4: [1.0]}


def _bits(x: np.ndarray) -> np.ndarray:
    t = torch.tensor(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _extreme_acts(tid: int, M: int, K: int) -> np.ndarray:
    """Unit-normal rows plus rows that drive the scales to their ends: zero, tiny (E4M3
    subnormal scales), large (E4M3 saturates at 448, codes saturate at 6), and a row whose
    halves differ by 2^40 (MXFP4 exponents far apart within a row)."""
    x = synth.bf16_bits_to_f32(make_acts(tid, M, K)).astype(np.float64)
    if M >= 6:
        x[0] = 0.0
        x[1] *= 1e-6
        x[2] *= 1e4
        x[3][: K // 2] *= 2.0 ** 40
        x[4][::3] = 0.0
        x[5] *= 1e-30
    return _bits(x)


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_quantize_act_bit_exact(fmt):
    for alpha in ALPHAS[fmt]:
        for M, K in ((1, 64), (7, 1024), (33, 992), (130, 5120)):
            if K % (16 if fmt == vt.NVFP4 else 32):
                continue
            A = _extreme_acts(synth.tensor_id(90, fmt, M, K), M, K)
            codes, scales = vt.quantize_act(bf16_dev(A), fmt, alpha)
            torch.cuda.synchronize()
            rc, rs, _ = oracle.quantize_act(fmt, A, alpha)
            assert np.array_equal(scales.cpu().numpy(), rs), (alpha, M, K)
            assert np.array_equal(codes.cpu().numpy(), rc), (alpha, M, K)


MIDPOINTS = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
EVEN_CODE = [0, 2, 2, 4, 4, 6, 6]  # E2M1 codes 0..7 = 0, .5, 1, 1.5, 2, 3, 4, 6: ties go to the even one


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_quantize_act_e2m1_midpoints(fmt):
    # every group holds 6 * 2^k (its largest magnitude), so the group step is exactly 2^k
    # (NVFP4 with alpha = 1: s = E4M3(2^k); MXFP4: e = k) and x / step lands exactly on each
    # midpoint of the E2M1 grid, on both signs, on its bf16 neighbours, on small magnitudes
    # that round to +0 from below zero, and on the saturation point
    g = 16 if fmt == vt.NVFP4 else 32
    vals = MIDPOINTS + [-v for v in MIDPOINTS]
    vals += [0.25 + 2 ** -9, 0.75 - 2 ** -8, 1.25 + 2 ** -7, 3.5 - 2 ** -6, -0.1, -0.2421875,
             0.0, 6.0, -6.0, 5.0 + 2 ** -5, -(2.5 - 2 ** -6)]
    per = g - 1
    groups = [vals[i:i + per] for i in range(0, len(vals), per)]
    rows = []
    for k in (0, -5, -8, 7):
        row = []
        for grp in groups:
            grp = grp + [0.0] * (per - len(grp))
            row += [6.0 * 2.0 ** k] + [v * 2.0 ** k for v in grp]
        rows.append(row)
    A = _bits(np.array(rows))
    M, K = A.shape
    codes, scales = vt.quantize_act(bf16_dev(A), fmt, 1.0)
    torch.cuda.synchronize()
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    rc, rs, _ = oracle.quantize_act(fmt, A, 1.0)
    assert np.array_equal(s, rs) and np.array_equal(c, rc)
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(M, K)
    for m in range(M):
        for j, v in enumerate(MIDPOINTS):  # the first group holds the midpoints, then their negatives
            assert nib[m, 1 + j] == EVEN_CODE[j], (m, v)
            neg = nib[m, 1 + len(MIDPOINTS) + j] if 1 + len(MIDPOINTS) + j < g else None
            if neg is not None:
                assert neg == (0 if EVEN_CODE[j] == 0 else 8 | EVEN_CODE[j]), (m, -v)


def test_quantize_act_strided_and_nonfinite():
    fmt, M, K = vt.NVFP4, 6, 256
    A = make_acts(synth.tensor_id(91, 0, 1), M, K)
    big = torch.zeros((M, K + 40), dtype=torch.bfloat16, device="cuda")
    big[:, :K] = bf16_dev(A)
    codes, scales = vt.quantize_act(big[:, :K], fmt, 0.05)
    rc, rs, _ = oracle.quantize_act(fmt, A, 0.05)
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    bad = A.copy()
    bad[2, 17] = 0x7F80  # +inf in group 1 of row 2
    bad[4, 200] = 0x7FC0  # NaN in group 12 of row 4
    for f, nan_byte in ((vt.NVFP4, 0x7F), (vt.MXFP4, 0xFF)):
        alpha = 0.05 if f == vt.NVFP4 else 1.0
        g = 16 if f == vt.NVFP4 else 32
        codes, scales = vt.quantize_act(bf16_dev(bad), f, alpha)
        c, s = codes.cpu().numpy(), scales.cpu().numpy()
        for (m, k) in ((2, 17), (4, 200)):
            j = k // g
            assert s[m, j] == nan_byte
            assert np.all(c[m, j * g // 2:(j + 1) * g // 2] == 0)
        rc, rs, _ = oracle.quantize_act(f, A, alpha)  # every other group as without the bad value
        mask = np.ones_like(rs, bool)
        mask[2, 17 // g] = mask[4, 200 // g] = False
        assert np.array_equal(s[mask], rs[mask])


SHAPES = [(128, 64), (640, 1024), (600, 992), (1000, 2048)]


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_w4a4_gemm_matches_oracle(fmt, N, K):
    if K % (16 if fmt == vt.NVFP4 else 32):
        pytest.skip("K not a multiple of the group")
    codes, scales, G = make_weight(fmt, synth.tensor_id(92, fmt, N, K), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    ws = W.new_workspace(300)
    for alpha in ALPHAS[fmt][:2]:
        for M in (1, 5, 16, 17, 128, 300):
            Ab = make_acts(synth.tensor_id(93, fmt, M, N + K), M, K)
            y = vt.w4a4_gemm(bf16_dev(Ab), W, alpha, workspace=ws)
            torch.cuda.synchronize()
            assert W.stats()["path"] == (1 if M <= 16 else 2)
            ref, _ = oracle.gemm_w4a4(fmt, Ab, alpha, codes, scales, G, N)
            check_rows(y.float().cpu().numpy(), ref, what=f"w4a4 fmt={fmt} a={alpha} M={M} N={N} K={K}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_w4a4_extreme_rows_both_paths(fmt):
    N, K = 384, 640
    codes, scales, G = make_weight(fmt, synth.tensor_id(94, fmt, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    alpha = 0.0078125 if fmt == vt.NVFP4 else 1.0
    for M, path in ((16, 1), (40, 2)):
        Ab = _extreme_acts(synth.tensor_id(94, fmt, 2, M), M, K)
        y = vt.w4a4_gemm(bf16_dev(Ab), W, alpha)
        torch.cuda.synchronize()
        assert W.stats()["path"] == path
        ref, _ = oracle.gemm_w4a4(fmt, Ab, alpha, codes, scales, G, N)
        got = y.float().cpu().numpy()
        assert np.all(got[0] == 0.0)
        check_rows(got, ref, what=f"extremes fmt={fmt} M={M}")


def test_w4a4_nonfinite_rows_give_nan_only_there():
    fmt, N, K = vt.NVFP4, 256, 512
    codes, scales, G = make_weight(fmt, synth.tensor_id(95, 0, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    for M in (4, 20):
        Ab = make_acts(synth.tensor_id(95, 0, 2, M), M, K)
        bad = Ab.copy()
        bad[1, 33] = 0x7F80
        y = vt.w4a4_gemm(bf16_dev(bad), W, 0.01).float().cpu().numpy()
        assert np.all(np.isnan(y[1]))
        keep = [m for m in range(M) if m != 1]
        ref, _ = oracle.gemm_w4a4(fmt, Ab[keep], 0.01, codes, scales, G, N)
        check_rows(y[keep], ref, what=f"nonfinite M={M}")


def test_w4a4_deterministic_and_grid_independent():
    fmt, N, K, M = vt.NVFP4, 1280, 1536, 260
    codes, scales, G = make_weight(fmt, synth.tensor_id(96, 0, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(96, 0, 2), M, K))
    first = vt.w4a4_gemm(A, W, 0.02).view(torch.int16).cpu()
    for opts in ({"grid": 1}, {"grid": 7}):
        again = vt.w4a4_gemm(A, W, 0.02, opts=opts).view(torch.int16).cpu()
        assert torch.equal(first, again), opts


def test_w4a4_rejections():
    fmt, N, K = vt.MXFP4, 128, 256
    codes, scales, G = make_weight(fmt, synth.tensor_id(97, 0, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(97, 0, 2), 4, K))
    with pytest.raises(vt.VtError):
        vt.w4a4_gemm(A, W, 0.5)  # MXFP4 activations have no global
    nc, ns, nG = make_weight(vt.NVFP4, synth.tensor_id(97, 0, 3), N, K)
    Wn = vt.PackedWeight.from_codes(to_dev(nc), to_dev(ns), nG, vt.NVFP4, N, K)
    for bad in (0.0, -1.0, float("nan"), float("inf"), 1e-40):
        with pytest.raises(vt.VtError):
            vt.w4a4_gemm(A, Wn, bad)
