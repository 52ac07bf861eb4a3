"""GPU: a seeded sweep of random shapes through every GEMM entry point against the oracle.

The fixed-shape tests pick shapes by hand; this one draws them (N from 1 to 3000, K any
multiple of the group up to 6144, M from 1 to 48 so that both the decode path and the tile
path run, with and without a row stride on A and C -- odd ones for C included -- from the
plain call, the greedy head and the W4A4 arm), so that no tile boundary, stage boundary or split-K range the hand-picked
shapes happen to avoid goes unchecked.  Every draw is fixed by its seed."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng(seed)
    fmt = int(rng.integers(0, 2))
    g = 16 if fmt == vt.NVFP4 else 32
    N = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(200, 3000))]))
    K = g * int(rng.integers(1, 6144 // g + 1))
    M = int(rng.choice([int(rng.integers(1, 17)), int(rng.integers(17, 49))]))
    pad_a = int(rng.choice([0, 8, 40]))
    pad_c = int(rng.choice([0, 1, 2, 31]))
    return fmt, N, K, M, pad_a, pad_c


@pytest.mark.parametrize("seed", range(24))
def test_random_shape_gemm(seed):
    fmt, N, K, M, pad_a, pad_c = _draw(seed)
    codes, scales, G = make_weight(fmt, synth.tensor_id(110, seed, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    Ab = make_acts(synth.tensor_id(110, seed, 2), M, K)
    A = torch.zeros((M, K + pad_a), dtype=torch.bfloat16, device="cuda")
    A[:, :K] = bf16_dev(Ab)
    C = torch.full((M, N + pad_c), 9.0, dtype=torch.bfloat16, device="cuda")  # any row stride
    vt.w4a16_gemm(A[:, :K], W, out=C[:, :N])
    torch.cuda.synchronize()
    assert W.stats()["path"] == (1 if M <= 16 else 2)
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    got = C.float().cpu().numpy()
    check_rows(got[:, :N], ref, what=f"seed={seed} fmt={fmt} N={N} K={K} M={M}")
    assert np.all(got[:, N:] == 9.0)  # the row padding of C is untouched


@pytest.mark.parametrize("seed", range(100, 108))
def test_random_shape_greedy(seed):
    fmt, N, K, M, _, _ = _draw(seed)
    M = min(M, 16)
    codes, scales, G = make_weight(fmt, synth.tensor_id(111, seed, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(111, seed, 2), M, K))
    tok, val = vt.w4a16_gemm_greedy(A, W)
    y = vt.w4a16_gemm(A, W)  # the plain output: the greedy choice is its first argmax
    torch.cuda.synchronize()
    yb = y.float().cpu().numpy()
    assert np.array_equal(tok.cpu().numpy(), np.argmax(yb, axis=1))
    assert np.array_equal(val.cpu().numpy(), yb[np.arange(M), np.argmax(yb, axis=1)])


@pytest.mark.parametrize("seed", range(200, 208))
def test_random_shape_w4a4(seed):
    fmt, N, K, M, _, _ = _draw(seed)
    alpha = 0.0078125 if fmt == vt.NVFP4 else 1.0
    codes, scales, G = make_weight(fmt, synth.tensor_id(112, seed, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    Ab = make_acts(synth.tensor_id(112, seed, 2), M, K)
    y = vt.w4a4_gemm(bf16_dev(Ab), W, alpha)
    torch.cuda.synchronize()
    ref, _ = oracle.gemm_w4a4(fmt, Ab, alpha, codes, scales, G, N)
    check_rows(y.float().cpu().numpy(), ref, what=f"w4a4 seed={seed} fmt={fmt} N={N} K={K} M={M}")
