"""CPU: the oracle's epilogue references -- the greedy token choice of the lm_head and the
SiLU-gated MLP input -- pinned against what their definitions and the mathematics fix:
constructed ties, NaN and signed-zero cases, numpy's first-occurrence argmax on finite
rows, the limits and the reflection identity of SiLU, exact bf16 rounding of halfway
values, linearity in the up half and the placement of the gate/up halves."""
import math

import numpy as np
import pytest

import oracle


def bits(values):
    """float -> bf16 bit patterns (every value used here is exactly representable)."""
    a = np.asarray(values, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# -------------------------------------------------------------------------- greedy
def test_greedy_ties_go_to_the_lowest_index():
    y = bits([[1.0, 2.0, 2.0, 1.0], [-3.0, -3.0, -3.0, -3.0], [0.5, 0.25, 0.5, 0.5]])
    idx, val = oracle.greedy(y)
    assert idx.tolist() == [1, 0, 0]
    assert val.tolist() == bits([2.0, -3.0, 0.5]).tolist()


def test_greedy_signed_zero_is_a_tie_and_nan_wins():
    zeros = np.array([[0x8000, 0x0000, bits([-1.0])[0]]], np.uint16)  # -0, +0, -1
    assert oracle.greedy(zeros)[0].tolist() == [0]
    nans = np.array([[bits([1.0])[0], 0x7FC0, bits([5.0])[0], 0x7FC0]], np.uint16)
    assert oracle.greedy(nans)[0].tolist() == [1]  # the first NaN
    ninf = np.array([[0xFF80, 0xFF80, 0xFF80]], np.uint16)  # all -inf
    assert oracle.greedy(ninf)[0].tolist() == [0]


def test_greedy_matches_first_occurrence_argmax_on_finite_rows():
    rng = np.random.default_rng(7)
    # a coarse grid forces many ties
    y = bits(np.round(rng.normal(size=(64, 1000)) * 4) / 4)
    idx, _ = oracle.greedy(y)
    ref = np.argmax(oracle.bf16_to_f32(y), axis=1)
    assert np.array_equal(idx, ref.astype(np.int32))


# ------------------------------------------------------------------------- silu*mul
def _silu_out(g, u):
    y = np.zeros((1, 2), np.float32)
    y[0, 0], y[0, 1] = g, u
    return int(oracle.silu_mul(y)[0, 0])


def test_silu_mul_limits():
    assert _silu_out(0.0, 3.0) == 0            # silu(0) = 0
    assert _silu_out(64.0, 0.5) == bits([32.0])[0]  # sigmoid(64) rounds to 1 in fp64
    v = oracle.bf16_to_f32(np.array([_silu_out(-40.0, 1.0)], np.uint16))[0]
    expect = -40.0 * math.exp(-40.0)           # silu(-40) ~ -40 e^-40, tiny but not zero
    assert v < 0 and abs(v / expect - 1) < 1e-2


def test_silu_reflection_identity():
    """silu(-x) = silu(x) - x, so (silu(x) - silu(-x)) * u = x * u."""
    for x in (0.5, 1.0, 2.75, 7.0):
        a = oracle.bf16_to_f32(np.array([_silu_out(x, 1.0)], np.uint16))[0]
        b = oracle.bf16_to_f32(np.array([_silu_out(-x, 1.0)], np.uint16))[0]
        assert abs((a - b) - x) <= 2 * 2 ** -8 * max(abs(a), abs(b), x)


def test_silu_mul_rounds_once_to_nearest_even():
    # silu(64) == 64 exactly, so the output is bf16(64 * u) with 64 * u exact in fp64
    assert _silu_out(64.0, (1 + 2 ** -8) * 2 ** -6) == bits([1.0])[0]              # tie -> even
    assert _silu_out(64.0, (1 + 3 * 2 ** -8) * 2 ** -6) == bits([1 + 2 ** -6])[0]  # tie -> even
    assert _silu_out(64.0, (1 + 2 ** -8 + 2 ** -20) * 2 ** -6) == bits([1 + 2 ** -7])[0]


def test_silu_mul_is_linear_in_up_and_reads_gate_then_up():
    rng = np.random.default_rng(3)
    I = 37
    y = rng.normal(size=(3, 2 * I)).astype(np.float32)
    out = oracle.silu_mul(y)
    y2 = y.copy()
    y2[:, I:] *= 4.0
    assert np.array_equal(oracle.bf16_to_f32(oracle.silu_mul(y2)), 4.0 * oracle.bf16_to_f32(out))
    swapped = np.concatenate([y[:, I:], y[:, :I]], axis=1)
    assert not np.array_equal(oracle.silu_mul(swapped), out)
    # gate <= -20 makes silu ~ 0 whatever the up half holds
    y3 = y.copy()
    y3[:, :I] = -20.0
    assert np.all(np.abs(oracle.bf16_to_f32(oracle.silu_mul(y3))) < 1e-6 * np.abs(y3[:, I:]).max() + 1e-30)
