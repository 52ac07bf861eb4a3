"""Pins for the oracle GEMM y = A . W^T (W dequantised), against exact rational arithmetic
on tiny inputs, closed forms for special cases, fp64 bounds and invariants.  The tests decode
bytes with the independently pinned tables (OCP E2M1 golden file, PyTorch E4M3/E8M0), never
with the oracle's own decoders."""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

import oracle
import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
E8M0 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def _bf16(x):
    t = torch.tensor(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def _pack(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _exact_weights(fmt, codes, sbytes, G):
    g = oracle.GROUP[fmt]
    mag = np.array(E2M1)[codes & 7]
    cv = np.where(codes & 8, -mag, mag)
    sv = (E4M3 if fmt == oracle.NVFP4 else E8M0)[sbytes]
    return cv * np.repeat(sv, g, axis=1) * G


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (2, 5, 64), (3, 8, 96), (3, 7, 128)])
def test_tiny_exact_gemm(fmt, M, N, K):
    """Small-integer A, power-of-two scales: every product and partial sum is exact in fp32,
    so the oracle must equal the exact rational result bit for bit."""
    rng = np.random.default_rng(M * 100 + N * 10 + K + fmt)
    g = oracle.GROUP[fmt]
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    if fmt == oracle.NVFP4:
        sb = rng.choice([0x30, 0x38, 0x40, 0x48], size=(N, K // g)).astype(np.uint8)  # 0.25..8
        G = 0.5
    else:
        sb = rng.integers(124, 131, size=(N, K // g)).astype(np.uint8)
        G = 1.0
    A = rng.integers(-8, 9, size=(M, K)).astype(np.float64)
    w = _exact_weights(fmt, codes, sb, G)
    exact = [[sum(Fraction(A[m, k]) * Fraction(w[n, k]) for k in range(K)) for n in range(N)]
             for m in range(M)]
    y, ybf = oracle.gemm(fmt, _bf16(A), _pack(codes), sb, G, N)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(y[m, n])) == exact[m][n]
    ref_bf = _bf16(np.array([[float(v) for v in r] for r in exact]))
    assert np.array_equal(ybf, ref_bf)


def test_unit_scales_reduce_to_e2m1_dot():
    """All scales 1.0 (E4M3 0x38, E8M0 0x7F) and G = 1: y = sum_k a_k * e2m1(c_k)."""
    rng = np.random.default_rng(5)
    M, N, K = 2, 4, 64
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    A = rng.integers(-4, 5, size=(M, K)).astype(np.float64)
    mag = np.array(E2M1)[codes & 7]
    cv = np.where(codes & 8, -mag, mag)
    want = A @ cv.T
    for fmt, sbyte in ((oracle.NVFP4, 0x38), (oracle.MXFP4, 0x7F)):
        sb = np.full((N, K // oracle.GROUP[fmt]), sbyte, np.uint8)
        y, _ = oracle.gemm(fmt, _bf16(A), _pack(codes), sb, 1.0, N)
        assert np.array_equal(y.astype(np.float64), want)


def test_all_ones_closed_form():
    """A all ones and every code c: y = K * c * s * G."""
    K, N = 256, 3
    for c, v in ((3, 1.5), (15, -6.0), (6, 4.0)):
        codes = np.full((N, K), c, np.uint8)
        sb = np.full((N, K // 16), 0x40, np.uint8)  # 2.0
        y, _ = oracle.gemm(oracle.NVFP4, _bf16(np.ones((1, K))), _pack(codes), sb, 0.25, N)
        assert np.all(y == K * v * 2.0 * 0.25)


def test_one_hot_selects_dequantised_column():
    N, K = 8, 128
    Wb = synth.normal_bf16(0, 77, 0.02, N, K)
    for fmt in (oracle.NVFP4, oracle.MXFP4):
        codes, scales, G = oracle.quantize(fmt, Wb)
        deq = oracle.dequant(fmt, codes, scales, G, N, K)
        A = np.zeros((K, K))
        A[np.arange(K), np.arange(K)] = 1.0
        y, _ = oracle.gemm(fmt, _bf16(A), codes, scales, G, N)
        assert np.array_equal(y, deq.T)


def test_dequant_matches_independent_decode():
    N, K = 16, 128
    Wb = synth.normal_bf16(0, 78, 0.02, N, K)
    codes, scales, G = oracle.quantize_nvfp4(Wb)
    c = np.zeros((N, K), np.uint8)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    w = _exact_weights(oracle.NVFP4, c, scales, 1.0)  # c*s exact
    want = (w.astype(np.float32) * np.float32(G)).astype(np.float32)
    got = oracle.dequant(oracle.NVFP4, codes, scales, G, N, K)
    assert np.array_equal(got, want)
    codes, scales = oracle.quantize_mxfp4(Wb)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    want = _exact_weights(oracle.MXFP4, c, scales, 1.0).astype(np.float32)
    assert np.array_equal(oracle.dequant(oracle.MXFP4, codes, scales, 1.0, N, K), want)


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_fp32_within_fp64_bound_and_invariants(fmt):
    M, N, K = 4, 24, 512
    Wb = synth.normal_bf16(0, 90 + fmt, 0.02, N, K)
    A = synth.normal_bf16(0, 91 + fmt, 1.0, M, K)
    codes, scales, G = oracle.quantize(fmt, Wb)
    y, _, y64 = oracle.gemm(fmt, A, codes, scales, G, N, want_f64=True)
    # recursive-summation bound: |fl(sum) - sum| <= K * u * sum|terms|, u = 2^-24
    deq = oracle.dequant(fmt, codes, scales, G, N, K).astype(np.float64)
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    absum = np.abs(a) @ np.abs(deq).T
    assert np.all(np.abs(y - y64) <= K * 2.0 ** -24 * absum)
    assert np.allclose(y64, a @ deq.T, rtol=1e-12, atol=1e-12)
    # sampled columns equal the full computation
    cols = [5, 0, 23, 5]
    ys, _ = oracle.gemm(fmt, A, codes, scales, G, N, cols=cols)
    assert np.array_equal(ys, y[:, cols])
    # permuting whole K-groups consistently in A and W changes y within rounding only
    g = oracle.GROUP[fmt]
    perm = np.random.default_rng(3).permutation(K // g)
    kperm = (perm[:, None] * g + np.arange(g)[None, :]).reshape(-1)
    c = np.zeros((N, K), np.uint8)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    yp, _ = oracle.gemm(fmt, A[:, kperm], _pack(c[:, kperm]), scales[:, perm], G, N)
    assert np.all(np.abs(yp - y) <= 2 * K * 2.0 ** -24 * absum)
    # linearity in A: y(2A) = 2 y(A) exactly (power-of-two scaling)
    A2 = _bf16(2 * a)
    y2, _ = oracle.gemm(fmt, A2, codes, scales, G, N)
    assert np.array_equal(y2, 2 * y)


def test_empty_batch():
    codes = np.zeros((4, 16), np.uint8)
    scales = np.full((4, 2), 0x38, np.uint8)
    y, ybf = oracle.gemm(oracle.NVFP4, np.zeros((0, 32), np.uint16), codes, scales, 1.0, 4)
    assert y.shape == (0, 4)


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_thread_count_changes_no_bit(fmt):
    """The oracle splits output columns (and weight rows) between threads; every output is
    still one sequential sum, so the thread count must not show in any bit."""
    M, N, K = 3, 37, 256
    Wb = synth.normal_bf16(0, 95 + fmt, 0.02, N, K)
    A = synth.normal_bf16(0, 96 + fmt, 1.0, M, K)
    q1 = oracle.quantize_nvfp4(Wb, nthreads=1) if fmt == oracle.NVFP4 else \
        oracle.quantize_mxfp4(Wb, nthreads=1)
    q5 = oracle.quantize_nvfp4(Wb, nthreads=5) if fmt == oracle.NVFP4 else \
        oracle.quantize_mxfp4(Wb, nthreads=5)
    for a, b in zip(q1, q5):
        assert np.array_equal(a, b)
    codes, scales = q1[:2]
    G = q1[2] if fmt == oracle.NVFP4 else 1.0
    ref = oracle.gemm(fmt, A, codes, scales, G, N, want_f64=True, nthreads=1)
    for t in (2, 5, 64):
        got = oracle.gemm(fmt, A, codes, scales, G, N, want_f64=True, nthreads=t)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b), t
