"""Pins for the oracle's synthetic-weight quantisers (NVFP4 and MXFP4).

Round trip: a tensor built from known codes and scales, with one +-6 code per group (so
the group's amax fixes its scale) and a power-of-two global, must quantise back to exactly
those bytes.  Error bound: each quantised weight lies within half a grid step (times the
group scale) of the input unless it saturated.  Scale choice: checked against the
definition with exact rationals."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def _codes_to_bytes(c: np.ndarray) -> np.ndarray:
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _code_values(c: np.ndarray) -> np.ndarray:
    mag = np.array(E2M1)[c & 7]
    return np.where(c & 8, -mag, mag)


@pytest.mark.parametrize("N,K", [(16, 64), (33, 160)])
def test_nvfp4_round_trip_exact(N, K):
    rng = np.random.default_rng(10)
    e4 = _e4m3_table()
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    codes[:, ::16] = rng.choice([7, 15], size=(N, K // 16))  # one +-6 per group
    # scales: any positive finite E4M3 byte; one group holds 448 so that amax = 6*448*G
    sb = rng.integers(0x08, 0x7E, size=(N, K // 16)).astype(np.uint8)
    sb[0, 0] = 0x7E
    G = 2.0 ** -12
    w = _code_values(codes) * np.repeat(e4[sb], 16, axis=1) * G
    Wb = _to_bf16_bits(w)
    assert np.array_equal(synth.bf16_bits_to_f32(Wb).astype(np.float64), w)  # exact in bf16
    qc, qs, qg = oracle.quantize_nvfp4(Wb)
    assert qg == G
    assert np.array_equal(qs, sb)
    # a code of -0 (8) decodes to the same value as +0 and is re-emitted as +0
    want = np.where(codes == 8, 0, codes).astype(np.uint8)
    assert np.array_equal(qc, _codes_to_bytes(want))


@pytest.mark.parametrize("N,K", [(16, 64), (9, 320)])
def test_mxfp4_round_trip_exact(N, K):
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    codes[:, ::32] = rng.choice([7, 15], size=(N, K // 32))
    eb = rng.integers(100, 140, size=(N, K // 32)).astype(np.uint8)
    w = _code_values(codes) * np.repeat(2.0 ** (eb.astype(np.float64) - 127), 32, axis=1)
    Wb = _to_bf16_bits(w)
    assert np.array_equal(synth.bf16_bits_to_f32(Wb).astype(np.float64), w)
    qc, qs = oracle.quantize_mxfp4(Wb)
    assert np.array_equal(qs, eb)
    want = np.where(codes == 8, 0, codes).astype(np.uint8)
    assert np.array_equal(qc, _codes_to_bytes(want))


def test_nvfp4_scale_and_error_bound_on_synthetic_weights():
    N, K = 64, 256
    Wb = synth.normal_bf16(0, 123, 0.02, N, K)
    w = synth.bf16_bits_to_f32(Wb).astype(np.float64)
    qc, qs, G = oracle.quantize_nvfp4(Wb)
    amax = np.abs(w).max()
    assert G == np.float32(amax / 2688.0)
    e4 = _e4m3_table()
    deq = oracle.dequant(oracle.NVFP4, qc, qs, G, N, K).astype(np.float64)
    for n in range(N):
        for g in range(K // 16):
            grp = w[n, g * 16:(g + 1) * 16]
            s = e4[qs[n, g]]
            # the scale byte is the E4M3 value nearest to amax_g / (6 G)
            target = Fraction(float(np.abs(grp).max())) / (6 * Fraction(float(G)))
            cands = [b for b in range(0x7F)]
            best = min(abs(Fraction(float(e4[b])) - target) for b in cands)
            assert abs(Fraction(float(s)) - target) == best
            step = 0.5 * s * G  # half the coarsest E2M1 gap (1.0 between 4 and 6 is 2x)
            err = np.abs(deq[n, g * 16:(g + 1) * 16] - grp)
            assert np.all(err <= 2 * step * (1 + 2 ** -20))


def test_mxfp4_error_bound_on_synthetic_weights():
    N, K = 32, 256
    Wb = synth.normal_bf16(0, 124, 0.02, N, K)
    w = synth.bf16_bits_to_f32(Wb).astype(np.float64)
    qc, qs = oracle.quantize_mxfp4(Wb)
    deq = oracle.dequant(oracle.MXFP4, qc, qs, 1.0, N, K).astype(np.float64)
    for n in range(N):
        for g in range(K // 32):
            grp = w[n, g * 32:(g + 1) * 32]
            scale = 2.0 ** (int(qs[n, g]) - 127)
            assert scale >= np.abs(grp).max() / 6 > scale / 2  # never clips
            err = np.abs(deq[n, g * 32:(g + 1) * 32] - grp)
            # gap between neighbours is at most 2 (4 -> 6), so error <= 1 * scale
            assert np.all(err <= scale)


def test_zero_group_and_zero_tensor():
    Z = np.zeros((4, 32), np.uint16)
    c, s, G = oracle.quantize_nvfp4(Z)
    assert G == 1.0 and not c.any() and not s.any()
    c, s = oracle.quantize_mxfp4(Z)
    assert not c.any() and np.all(s == 0)  # e = -127 -> byte 0


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize_nvfp4(np.zeros((4, 24), np.uint16))
    with pytest.raises(ValueError):
        oracle.quantize_mxfp4(np.zeros((4, 48), np.uint16))
