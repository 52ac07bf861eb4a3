"""CPU pins of the oracle's W4A4 arm (activation quantiser + GEMM on the dequantised
activations), each against something other than the oracle itself: groups worked out by
hand (golden file), exact reconstruction of activations that already lie on the FP4 grid
(where the W4A4 layer must equal the independently pinned W4A16 layer bit for bit), a brute
force nearest-point search over the E2M1 and E4M3 grids in fp64, sign and power-of-two
symmetries, and the rejections."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w4a4_act_quant_worked.txt")
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _bf16_bits(x) -> np.ndarray:
    t = torch.tensor(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ") if line.startswith("case") else line.partition(":")
        if key == "case":
            fmt, alpha = rest.split()
            cur = {"fmt": oracle.NVFP4 if fmt == "nvfp4" else oracle.MXFP4, "alpha": float(alpha)}
            cases.append(cur)
        elif key == "x":
            cur["x"] = [float(v) for v in rest.split()]
        elif key == "scale":
            cur["scale"] = int(rest.strip(), 16)
        elif key == "codes":
            cur["codes"] = [int(v, 16) for v in rest.split()]
        elif key == "deq":
            cur["deq"] = [float(v) for v in rest.split()]
    return cases


def _nibbles(codes: np.ndarray) -> np.ndarray:
    """[M, K/2] packed bytes -> [M, K] codes (low nibble = even k)."""
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def _e2m1_val(c: np.ndarray) -> np.ndarray:
    v = E2M1[c & 7]
    return np.where(c & 8, -v, v)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"fmt{c['fmt']}_a{c['alpha']}")
def test_worked_groups_golden(case):
    g = 16 if case["fmt"] == oracle.NVFP4 else 32
    x = np.zeros(g)
    x[: len(case["x"])] = case["x"]
    bits = _bf16_bits(x)[None, :]
    assert np.array_equal(oracle.bf16_to_f32(bits)[0], x.astype(np.float32)), "inputs bf16-exact"
    codes, scales, aq = oracle.quantize_act(case["fmt"], bits, case["alpha"])
    want_codes = np.zeros(g, np.uint8)
    want_codes[: len(case["codes"])] = case["codes"]
    want_deq = np.zeros(g)
    want_deq[: len(case["deq"])] = case["deq"]
    assert scales[0, 0] == case["scale"]
    assert np.array_equal(_nibbles(codes)[0], want_codes)
    assert np.array_equal(aq[0].astype(np.float64), want_deq)


def _on_grid_nv(rng, M, K, alpha_exp):
    """Activations c * s * 2^alpha_exp exactly (bf16), each group holding a +-6 s element so
    that its scale is recovered exactly."""
    g = 16
    c = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    c[(c & 7) == 0] = 0  # canonical zero
    sbytes = rng.integers(0x20, 0x70, size=(M, K // g)).astype(np.uint8)  # normal E4M3
    lead = rng.integers(0, g, size=(M, K // g))
    for m in range(M):
        for j in range(K // g):
            c[m, j * g + lead[m, j]] = 7 | (8 if rng.random() < 0.5 else 0)
    s = np.array([oracle.e4m3_value(int(b)) for b in sbytes.ravel()]).reshape(sbytes.shape)
    x = _e2m1_val(c) * np.repeat(s, g, axis=1) * 2.0 ** alpha_exp
    return x, c, sbytes


def test_on_grid_nvfp4_recovered_and_equals_w4a16():
    rng = np.random.default_rng(11)
    M, K, N = 5, 256, 48
    for alpha_exp in (-7, 0, 3):
        x, c, sbytes = _on_grid_nv(rng, M, K, alpha_exp)
        A = _bf16_bits(x)
        assert np.array_equal(oracle.bf16_to_f32(A).astype(np.float64), x)
        codes, scales, aq = oracle.quantize_act(oracle.NVFP4, A, 2.0 ** alpha_exp)
        assert np.array_equal(scales, sbytes)
        assert np.array_equal(_nibbles(codes), c)
        assert np.array_equal(aq.astype(np.float64), x)
        # the layer on on-grid activations is the W4A16 layer on the same bf16 values
        W = synth.normal_bf16(3, 40 + alpha_exp, 0.02, N, K)
        wc, ws, G = oracle.quantize(oracle.NVFP4, W)
        y4, b4 = oracle.gemm_w4a4(oracle.NVFP4, A, 2.0 ** alpha_exp, wc, ws, G, N)
        y16, b16 = oracle.gemm(oracle.NVFP4, A, wc, ws, G, N)
        assert np.array_equal(y4, y16) and np.array_equal(b4, b16)


def test_on_grid_mxfp4_recovered_and_equals_w4a16():
    rng = np.random.default_rng(12)
    M, K, N, g = 4, 256, 40, 32
    c = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    c[(c & 7) == 0] = 0
    e = rng.integers(-20, 20, size=(M, K // g))
    for m in range(M):
        for j in range(K // g):
            c[m, j * g + rng.integers(0, g)] = 7 | (8 if rng.random() < 0.5 else 0)
    x = _e2m1_val(c) * np.repeat(2.0 ** e, g, axis=1)
    A = _bf16_bits(x)
    codes, scales, aq = oracle.quantize_act(oracle.MXFP4, A)
    assert np.array_equal(scales.astype(np.int64), e + 127)
    assert np.array_equal(_nibbles(codes), c)
    assert np.array_equal(aq.astype(np.float64), x)
    W = synth.normal_bf16(3, 50, 0.02, N, K)
    wc, ws, G = oracle.quantize(oracle.MXFP4, W)
    y4, _ = oracle.gemm_w4a4(oracle.MXFP4, A, 1.0, wc, ws, G, N)
    y16, _ = oracle.gemm(oracle.MXFP4, A, wc, ws, G, N)
    assert np.array_equal(y4, y16)


E4M3_POS = np.array([oracle.e4m3_value(b) for b in range(0x7F)])  # 0 .. 448


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_nearest_point_brute_force(fmt):
    """Every code is a nearest point of the scaled E2M1 grid (saturating), and every NVFP4
    scale a nearest E4M3 value to amax / (6 alpha), by exhaustive search in fp64; a decision
    may differ from the exact real one only where the two candidates are equally near to
    within the fp32 rounding of the quotient."""
    g = 16 if fmt == oracle.NVFP4 else 32
    alpha = 0.0078125 if fmt == oracle.NVFP4 else 1.0
    A = synth.normal_bf16(5, 60 + fmt, 1.0, 24, 512)
    x = oracle.bf16_to_f32(A).astype(np.float64)
    codes, scales, aq = oracle.quantize_act(fmt, A, alpha)
    c = _nibbles(codes)
    M, K = x.shape
    for m in range(M):
        for j in range(K // g):
            xs = x[m, j * g:(j + 1) * g]
            amax = np.abs(xs).max()
            if fmt == oracle.NVFP4:
                q = amax / (6 * alpha)
                d = np.abs(E4M3_POS - min(q, 448.0))
                sb = int(scales[m, j])
                assert d[sb] <= d.min() * (1 + 1e-6) + 1e-30, (m, j, q, sb)
                step = E4M3_POS[sb] * alpha
            else:
                step = 2.0 ** (int(scales[m, j]) - 127)
                assert 6 * step >= amax and (amax == 0 or 3 * step < amax)
            if step == 0:
                assert np.all(c[m, j * g:(j + 1) * g] == 0)
                continue
            for i in range(g):
                r = xs[i] / step
                dist = np.abs(E2M1 - min(abs(r), 6.0))
                got = int(c[m, j * g + i])
                assert dist[got & 7] <= dist.min() + 1e-6 * max(1.0, abs(r)), (m, j, i, r, got)
                if got & 7:
                    assert (got >> 3) == (1 if r < 0 else 0)
                if fmt == oracle.NVFP4:
                    cs = np.float32(_e2m1_val(np.uint8(got)) * E4M3_POS[sb])
                    want = np.float32(cs * np.float32(alpha))
                else:
                    want = _e2m1_val(np.uint8(got)) * step
                assert aq[m, j * g + i] == want


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_sign_and_power_of_two_symmetry(fmt):
    A = synth.normal_bf16(6, 70 + fmt, 1.0, 16, 256)
    alpha = 0.03125 if fmt == oracle.NVFP4 else 1.0
    c0, s0, q0 = oracle.quantize_act(fmt, A, alpha)
    neg = A ^ np.uint16(0x8000)
    c1, s1, q1 = oracle.quantize_act(fmt, neg, alpha)
    n0, n1 = _nibbles(c0), _nibbles(c1)
    assert np.array_equal(s0, s1)
    assert np.array_equal(n1, np.where(n0 & 7, n0 ^ 8, 0))
    assert np.array_equal(q1, -q0 + 0.0)
    # scaling by 2^j (bf16 exponent field, no subnormals here) moves only the scales
    j = 5
    up = _bf16_bits(oracle.bf16_to_f32(A).astype(np.float64) * 2.0 ** j)
    if fmt == oracle.NVFP4:
        c2, s2, q2 = oracle.quantize_act(fmt, up, alpha * 2.0 ** j)
        assert np.array_equal(s2, s0)
    else:
        c2, s2, q2 = oracle.quantize_act(fmt, up)
        assert np.array_equal(s2.astype(int), s0.astype(int) + j)
    assert np.array_equal(c2, c0)
    assert np.array_equal(q2.astype(np.float64), q0.astype(np.float64) * 2.0 ** j)


def test_rejections():
    A = synth.normal_bf16(7, 80, 1.0, 2, 64)
    for alpha in (0.0, -1.0, float("nan"), float("inf"), 1e-40):
        with pytest.raises(ValueError):
            oracle.quantize_act(oracle.NVFP4, A, alpha)
    with pytest.raises(ValueError):
        oracle.quantize_act(oracle.MXFP4, A, 0.5)
    bad = A.copy()
    bad[1, 3] = 0x7F80  # +inf
    with pytest.raises(ValueError):
        oracle.quantize_act(oracle.NVFP4, bad, 1.0)
    with pytest.raises(ValueError):
        oracle.quantize_act(oracle.MXFP4, A[:, :48])  # K not a multiple of 32
