"""CPU: the seeded input generator against its published definition.  Both sides of every
parity test draw their inputs here, so a generator that silently changed (or threaded its
rows differently) would move every fixture at once; these checks restate the definition
(SplitMix64, Steele, Lea and Flood 2014; Box-Muller) in plain Python integers and floats."""
import math

import numpy as np
import torch

import synth

MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _mix64(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_splitmix64_published_outputs():
    """The first outputs of SplitMix64 started from state 0."""
    assert _mix64(GAMMA) == 0xE220A8397B1DCDAF
    assert _mix64((2 * GAMMA) & MASK) == 0x6E789E6AA1B965F4
    assert _mix64((3 * GAMMA) & MASK) == 0x06C45D188009454F


def _element(seed, tid, sigma, i):
    base = _mix64((seed * GAMMA + tid) & MASK)
    j = i >> 1
    x1 = _mix64((base + (2 * j + 1) * GAMMA) & MASK)
    x2 = _mix64((base + (2 * j + 2) * GAMMA) & MASK)
    u1 = ((x1 >> 11) + 1) * 2.0 ** -53
    u2 = (x2 >> 11) * 2.0 ** -53
    r = math.sqrt(-2.0 * math.log(u1))
    z = r * (math.sin(2 * math.pi * u2) if i & 1 else math.cos(2 * math.pi * u2))
    return sigma * z


def _bf16_bits(x):
    return int(torch.tensor([x], dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
               .view(torch.int16).numpy().astype(np.uint16)[0])


def test_elements_follow_the_definition():
    seed, tid, sigma, rows, cols = 3, synth.tensor_id(7, 2, synth.ROLE_W, 5), 0.02, 5, 37
    got = synth.normal_bf16(seed, tid, sigma, rows, cols)
    for i in list(range(12)) + [36, 37, 100, rows * cols - 1]:
        assert int(got.reshape(-1)[i]) == _bf16_bits(_element(seed, tid, sigma, i)), i


def test_rows_regenerate_alone_and_ids_are_independent():
    seed, tid, cols = 0, synth.tensor_id(2, 0, synth.ROLE_A), 96
    full = synth.normal_bf16(seed, tid, 1.0, 40, cols)
    pick = [39, 0, 17, 17]
    assert np.array_equal(synth.normal_bf16_rows(seed, tid, 1.0, cols, pick), full[pick])
    other = synth.normal_bf16(seed, tid + 1, 1.0, 40, cols)
    assert np.mean(other == full) < 0.05
    assert synth.normal_bf16(seed, tid, 1.0, 0, cols).shape == (0, cols)


def test_moments_match_the_normal_law():
    x = synth.bf16_bits_to_f32(synth.normal_bf16(1, 99, 0.02, 256, 1024)).astype(np.float64)
    n = x.size
    assert abs(x.mean()) < 5 * 0.02 / math.sqrt(n)
    assert abs(x.std() / 0.02 - 1.0) < 0.01
    assert abs(np.mean(np.abs(x) < 0.02) - 0.6827) < 0.01  # one-sigma mass
