"""Pins for the oracle's format decoders and rounding, against things other than itself:
the OCP E2M1 table (golden file), PyTorch's float8_e4m3fn / float8_e8m0fnu dtypes (an
independent library decode of every byte), exact rational arithmetic, and invariants."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()[:2]
        rows.append((a, b))
    return rows


def test_e2m1_table_matches_ocp_golden():
    rows = _read_pairs("e2m1_table.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_value(int(code))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_decode_all_bytes_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        got = oracle.e4m3_value(b)
        want = ref[b].item()
        if math.isnan(want):
            assert math.isnan(got), b
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (b, got, want)


def test_e4m3_anchors_and_invariants():
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    vals = [oracle.e4m3_value(b) for b in range(0x7F)]
    assert all(vals[i] < vals[i + 1] for i in range(len(vals) - 1))  # monotonic 0x00..0x7E
    for b in range(0x7F):
        assert oracle.e4m3_value(b | 0x80) == -oracle.e4m3_value(b)
    assert max(vals) == 448.0


def test_e8m0_decode_all_bytes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for b in range(256):
        got = oracle.e8m0_value(b)
        if b == 0xFF:
            assert math.isnan(got) and math.isnan(ref[b].item())
            continue
        assert got == ref[b].item() == 2.0 ** (b - 127), b
    assert oracle.e8m0_value(0x7F) == 1.0


def test_e2m1_rounding_ties_golden():
    for q, code in _read_pairs("e2m1_round_ties.txt"):
        assert oracle.e2m1_from_real(float(q)) == int(code), q


def test_e2m1_rounding_is_nearest_on_a_grid():
    # brute force: the chosen value is never farther than any other representable value
    table = [Fraction(v) for _, v in _read_pairs("e2m1_table.txt")][:8]
    for i in range(-1400, 1401):
        q = i / 200.0
        c = oracle.e2m1_from_real(q)
        mag = c & 7
        chosen = table[mag] * (-1 if (c & 8) else 1)
        best = min(abs(Fraction(q) - t * s) for t in table for s in (1, -1)
                   if abs(t) <= 6)
        if abs(q) <= 6:
            assert abs(Fraction(q) - chosen) == best, (q, c)
        else:
            assert mag == 7 and ((c & 8) != 0) == (q < 0)


def test_e4m3_rounding_matches_torch_below_448():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.uniform(0, 448, 4000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 4000)),
        [oracle.e4m3_value(b) for b in range(0x7F)],
        # exact midpoints between neighbours: the tie rule decides
        [(oracle.e4m3_value(b) + oracle.e4m3_value(b + 1)) / 2 for b in range(0x7E)],
    ])
    xs = xs[xs < 448.0]
    ref = torch.tensor(xs, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8)
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert oracle.e4m3_from_real(x) == r, x


def test_e4m3_rounding_saturates():
    for x in (448.0, 450.0, 464.0, 479.0, 1e6, math.inf):
        assert oracle.e4m3_from_real(x) == 0x7E


def test_mx_exponent_is_smallest_power_of_two_bound():
    rng = np.random.default_rng(1)
    vals = list(np.exp(rng.uniform(np.log(1e-30), np.log(1e30), 3000))) + \
        [6.0 * 2.0 ** k for k in range(-40, 40)] + [3.0, 6.0, 12.0, 0.75, 1e-38]
    for a in vals:
        e = oracle.mx_exponent(float(a))
        A = Fraction(float(a)) / 6
        assert Fraction(2) ** e >= A, (a, e)
        if e > -127:  # -127 is the clamp floor
            assert Fraction(2) ** (e - 1) < A, (a, e)
        else:
            assert A <= Fraction(2) ** -127
    assert oracle.mx_exponent(0.0) == -127
    assert oracle.mx_exponent(1e-45) == -127  # clamped


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 100,
                         (np.arange(1, 4000, dtype=np.uint32) * 0x8000 + 0x3F800000).view(np.float32)])
    ref = torch.tensor(xs, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert oracle.f32_to_bf16(x) == r, x
