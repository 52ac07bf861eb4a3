"""GPU: repeated runs give the same bits.  Every output element of the decode and grouped
(mixture-of-experts) kernels is a fixed-order sum for a given launch shape, so any run-to-run
change is a hand-off race between the kernels' roles (producer, consumers, publisher,
reducer), the kind that a single comparison catches only some of the time.  Each launch
shape is run many times, with the ring stages reused many times over (few CTAs)."""
import numpy as np
import pytest
import torch

import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu

REPS = 10


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_repeats_bit_for_bit(fmt, M):
    N, K = 2048, 3072
    codes, scales, G = make_weight(fmt, synth.tensor_id(120, fmt, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    A = bf16_dev(make_acts(synth.tensor_id(120, fmt, 2, M), M, K))
    ws = W.new_workspace(16)
    for opts in (None, {"grid": 1}, {"grid": 3}, {"grid": 64}, {"force_path": 3}):
        first = vt.w4a16_gemm(A, W, workspace=ws, opts=opts).view(torch.int16).clone()
        for r in range(REPS):
            again = vt.w4a16_gemm(A, W, workspace=ws, opts=opts).view(torch.int16)
            assert torch.equal(first, again), (opts, r)
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_moe_repeats_bit_for_bit(fmt):
    E, N, K, topk = 16, 768, 1024, 4
    srcs = [make_weight(fmt, synth.tensor_id(121, fmt, e), N, K) for e in range(E)]
    W = vt.PackedWeight.grouped(to_dev(np.stack([s[0] for s in srcs])),
                                to_dev(np.stack([s[1] for s in srcs])), [s[2] for s in srcs],
                                fmt, E, N, K)
    rng = np.random.default_rng(7)
    for M in (1, 6, 16):
        ids = to_dev(np.stack([rng.choice(E, size=topk, replace=False)
                               for _ in range(M)]).astype(np.int32))
        A = bf16_dev(make_acts(synth.tensor_id(121, fmt, 99, M), M, K))
        ws = W.moe_workspace(M, topk)
        first = vt.w4a16_gemm_moe(A, W, ids, workspace=ws).view(torch.int16).clone()
        for r in range(REPS):
            again = vt.w4a16_gemm_moe(A, W, ids, workspace=ws).view(torch.int16)
            assert torch.equal(first, again), (M, r)
        assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_silu_and_greedy_repeat_bit_for_bit(fmt):
    I, K = 1024, 2048
    dev = lambda t: (to_dev(t[0]), to_dev(t[1]), t[2])
    g = make_weight(fmt, synth.tensor_id(122, fmt, synth.ROLE_GATE), I, K)
    u = make_weight(fmt, synth.tensor_id(122, fmt, synth.ROLE_UP), I, K)
    Wp = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K, paired=True)
    for M in (2, 12, 40):
        A = bf16_dev(make_acts(synth.tensor_id(122, fmt, 3, M), M, K))
        first = vt.w4a16_gemm_silu_mul(A, Wp).view(torch.int16).clone()
        tok0 = vt.w4a16_gemm_greedy(A[:min(M, 16)], Wp)[0].clone()
        for r in range(REPS):
            assert torch.equal(first, vt.w4a16_gemm_silu_mul(A, Wp).view(torch.int16)), (M, r)
            assert torch.equal(tok0, vt.w4a16_gemm_greedy(A[:min(M, 16)], Wp)[0]), (M, r)
