"""GPU: the fused MLP decode (vt_fp4_w4a16_mlp): down(silu(gate) * up) in one GEMM kernel.

Checked against the oracle's chain (fp32 gate and up sums, silu(g) * u in fp64 rounded once
to bf16, then the down GEMM on those bf16 activations) with the GEMM tolerance, across several
tiles with ragged I, N and K, every M of the decode path; against the two separate calls
(vt_fp4_w4a16_gemm_silu_mul, then vt_fp4_w4a16_gemm) bit for bit at the MXFP4 MLP workload's
full size, where both run on the same grid; repeated and graph-captured calls (the grid
barrier's generation carries from call to call); the bounded-wait failure path; rejections."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _mlp(fmt, I, K, N, tag):
    g = make_weight(fmt, synth.tensor_id(70, tag, synth.ROLE_GATE), I, K)
    u = make_weight(fmt, synth.tensor_id(70, tag, synth.ROLE_UP), I, K)
    d = make_weight(fmt, synth.tensor_id(70, tag, 13), N, I)
    dev = lambda t: (to_dev(t[0]), to_dev(t[1]), t[2])
    Wg = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K, paired=True)
    Wd = vt.PackedWeight.from_codes(to_dev(d[0]), to_dev(d[1]), d[2], fmt, N, I)
    return g, u, d, Wg, Wd


def _oracle_chain(fmt, Ab, g, u, d, I, N):
    yg, _ = oracle.gemm(fmt, Ab, g[0], g[1], g[2], I)
    yu, _ = oracle.gemm(fmt, Ab, u[0], u[1], u[2], I)
    act = oracle.silu_mul(np.concatenate([yg, yu], axis=1))  # bf16 bits [M, I]
    y, _ = oracle.gemm(fmt, act, d[0], d[1], d[2], N)
    return oracle.bf16_to_f32(act), y


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("I,K,N", [(96, 512, 200), (640, 1024, 384), (992, 2048, 1100)])
def test_fused_mlp_matches_oracle(fmt, I, K, N):
    if I % (16 if fmt == vt.NVFP4 else 32):
        pytest.skip("the down projection's K = I must be a multiple of the group")
    g, u, d, Wg, Wd = _mlp(fmt, I, K, N, I)
    ws = vt.mlp_workspace(Wg, Wd)
    for M in (1, 2, 5, 8, 9, 16):
        Ab = make_acts(synth.tensor_id(71, fmt, I, M), M, K)
        act = torch.full((M, I), 7.0, dtype=torch.bfloat16, device="cuda")
        y = vt.w4a16_mlp(bf16_dev(Ab), Wg, Wd, act=act, workspace=ws)
        torch.cuda.synchronize()
        assert Wd.stats()["launches"] == 2
        ref_act, ref_y = _oracle_chain(fmt, Ab, g, u, d, I, N)
        check_rows(act.float().cpu().numpy(), ref_act, what=f"act fmt={fmt} I={I} M={M}")
        check_rows(y.float().cpu().numpy(), ref_y, what=f"mlp fmt={fmt} I={I} K={K} N={N} M={M}")
    assert vt.workspace_status(ws) == 0


def test_fused_mlp_without_act_output_and_strided():
    fmt, I, K, N, M = vt.MXFP4, 640, 1024, 384, 6
    g, u, d, Wg, Wd = _mlp(fmt, I, K, N, 1)
    Ab = make_acts(synth.tensor_id(72, 1, 0), M, K)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :K] = bf16_dev(Ab)
    out = torch.full((M, N + 10), 5.0, dtype=torch.bfloat16, device="cuda")
    vt.w4a16_mlp(big[:, :K], Wg, Wd, out=out[:, :N])
    torch.cuda.synchronize()
    _, ref_y = _oracle_chain(fmt, Ab, g, u, d, I, N)
    o = out.float().cpu().numpy()
    check_rows(o[:, :N], ref_y, what="strided, no act")
    assert np.all(o[:, N:] == 5.0)


def test_fused_mlp_repeated_and_in_a_graph():
    """Calls of several M back to back on one workspace, eagerly and replayed from a graph:
    every replay gives the first run's bits and the status word stays clear."""
    fmt, I, K, N = vt.NVFP4, 992, 2048, 1100
    g, u, d, Wg, Wd = _mlp(fmt, I, K, N, 2)
    ws = vt.mlp_workspace(Wg, Wd)
    Ms = [1, 4, 16, 3, 8]
    A = [bf16_dev(make_acts(synth.tensor_id(73, M, 0), M, K)) for M in Ms]
    Y = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for M in Ms]
    s = torch.cuda.Stream()

    def issue():
        for a, y in zip(A, Y):
            vt.w4a16_mlp(a, Wg, Wd, out=y, workspace=ws, stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        issue()
    s.synchronize()
    first = [y.clone() for y in Y]
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        issue()
    for _ in range(3):
        for y in Y:
            y.fill_(0)
        with torch.cuda.stream(s):
            gr.replay()
        s.synchronize()
        for y, f in zip(Y, first):
            assert torch.equal(y.view(torch.int16), f.view(torch.int16))
    for M, a, f in zip(Ms, A, first):
        Ab = a.view(torch.int16).cpu().numpy().view(np.uint16)
        _, ref_y = _oracle_chain(fmt, Ab, g, u, d, I, N)
        check_rows(f.float().cpu().numpy(), ref_y, what=f"graph M={M}")
    assert vt.workspace_status(ws) == 0


def test_fused_mlp_equals_the_two_calls_at_full_size():
    """The MXFP4 MLP workload's shapes (gate_up 2 x 12288 x 4096, down 4096 x 12288): both
    GEMMs have enough work for one CTA per SM, so the fused kernel and the two separate calls
    split the work identically and must agree bit for bit, act and output."""
    fmt, I, K, N = vt.MXFP4, 12288, 4096, 4096
    gen = torch.Generator(device="cuda").manual_seed(5)

    def rand_weight(rows, cols):
        codes = torch.randint(0, 256, (rows, cols // 2), dtype=torch.uint8, device="cuda",
                              generator=gen)
        scales = torch.randint(118, 124, (rows, cols // 32), dtype=torch.uint8, device="cuda",
                               generator=gen)
        return codes, scales, 1.0

    Wg = vt.PackedWeight.gate_up(rand_weight(I, K), rand_weight(I, K), fmt, I, K, paired=True)
    Wd = vt.PackedWeight.from_codes(*rand_weight(N, I), fmt, N, I)
    ws = vt.mlp_workspace(Wg, Wd)
    ws2 = Wg.new_workspace(16)
    ws3 = Wd.new_workspace(16)
    for M in (1, 2, 4, 8, 16):
        A = torch.randn((M, K), device="cuda", generator=gen).to(torch.bfloat16)
        act = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
        y = vt.w4a16_mlp(A, Wg, Wd, act=act, workspace=ws)
        act2 = vt.w4a16_gemm_silu_mul(A, Wg, workspace=ws2)
        y2 = vt.w4a16_gemm(act2, Wd, workspace=ws3)
        torch.cuda.synchronize()
        assert torch.equal(act.view(torch.int16), act2.view(torch.int16)), M
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), M
    assert vt.workspace_status(ws) == 0


def test_fused_mlp_bounded_waits_time_out_and_recover():
    fmt, I, K, N, M = vt.NVFP4, 640, 2048, 640, 4
    g, u, d, Wg, Wd = _mlp(fmt, I, K, N, 3)
    ws = vt.mlp_workspace(Wg, Wd)
    Ab = make_acts(synth.tensor_id(74, 1, 0), M, K)
    A = bf16_dev(Ab)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    vt.w4a16_mlp(A, Wg, Wd, workspace=ws, opts={"withhold_weights": 1, "wait_limit_us": 20000})
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.5
    assert vt.workspace_status(ws) == _lib.VT_ERR_TIMEOUT
    assert vt.workspace_status(ws) == _lib.VT_OK
    y = vt.w4a16_mlp(A, Wg, Wd, workspace=ws)
    torch.cuda.synchronize()
    _, ref_y = _oracle_chain(fmt, Ab, g, u, d, I, N)
    check_rows(y.float().cpu().numpy(), ref_y, what="after timeout")
    assert vt.workspace_status(ws) == _lib.VT_OK


def test_fused_mlp_rejections():
    fmt, I, K, N = vt.NVFP4, 128, 256, 128
    g, u, d, Wg, Wd = _mlp(fmt, I, K, N, 4)
    Ws = vt.PackedWeight.gate_up((to_dev(g[0]), to_dev(g[1]), g[2]),
                                 (to_dev(u[0]), to_dev(u[1]), u[2]), fmt, I, K)  # not paired
    A = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    bad_cases = [
        lambda: vt.w4a16_mlp(A, Ws, Wd),                                   # gate_up not paired
        lambda: vt.w4a16_mlp(A, Wg, Wg),                                   # down paired
        lambda: vt.w4a16_mlp(torch.zeros((17, K), dtype=torch.bfloat16, device="cuda"), Wg, Wd),
        lambda: vt.w4a16_mlp(A, Wg, Wd, opts={"grid": 100000}),           # more CTAs than SMs
        lambda: vt.w4a16_mlp(A, Wg, Wd, opts={"warps": 4}),
        lambda: vt.w4a16_mlp(A, Wg, Wd, opts={"force_path": 2}),
    ]
    dm = make_weight(fmt, synth.tensor_id(70, 9, 13), N, 2 * I)
    Wk = vt.PackedWeight.from_codes(to_dev(dm[0]), to_dev(dm[1]), dm[2], fmt, N, 2 * I)
    bad_cases.append(lambda: vt.w4a16_mlp(A, Wg, Wk))                      # down K != I
    dx = make_weight(vt.MXFP4, synth.tensor_id(70, 10, 13), N, I)
    Wx = vt.PackedWeight.from_codes(to_dev(dx[0]), to_dev(dx[1]), dx[2], vt.MXFP4, N, I)
    bad_cases.append(lambda: vt.w4a16_mlp(A, Wg, Wx))                      # formats differ
    for i, call in enumerate(bad_cases):
        with pytest.raises(_lib.VtError) as e:
            call()
        assert e.value.status == _lib.VT_ERR_INVALID_ARG, i
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.VtError):
        vt.w4a16_mlp(A, Wg, Wd, workspace=small)
    assert vt.w4a16_mlp(A[:0], Wg, Wd).shape == (0, N)
