"""GPU: the per-group tile epilogue of the decode kernel.  For up to 2 tokens, when a CTA
covers at least three 128-row tiles (the lm_head-like calls), the library launches a decode
kernel in which a complete tile's rows are summed per row-block group by one of its warps in
turn, instead of after two CTA-wide barriers; the sums and their order are unchanged.  These
tests reach it at small sizes -- by a 2-CTA launch shape, or by a weight of many row tiles
under the default launch shape -- on the plain, fused gate_up (two globals) and paired
layouts and through the greedy head, against the oracle; the same launch shape twice gives
the same bits."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, bf16_host_bits, check_rows, make_acts, make_weight, to_dev
from test_gpu_greedy import _first_argmax, check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_plain_fused_and_paired_weights_on_two_ctas(fmt):
    # 2 CTAs: plain 1000 x 1024 is 8 row tiles (ragged) of 16 k tiles, 4 per CTA; the fused
    # gate_up of I = 700 is 11 row tiles, 5.5 per CTA (the middle tile is shared)
    N, K, I = 1000, 1024, 700
    c, s, G = make_weight(fmt, synth.tensor_id(87, fmt, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(c), to_dev(s), G, fmt, N, K)
    g = make_weight(fmt, synth.tensor_id(87, fmt, synth.ROLE_GATE), I, K)
    u = make_weight(fmt, synth.tensor_id(87, fmt, synth.ROLE_UP), I, K)
    dev = lambda t: (to_dev(t[0]), to_dev(t[1]), t[2])
    Wf = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K)
    Wp = vt.PackedWeight.gate_up(dev(g), dev(u), fmt, I, K, paired=True)
    for M in (1, 2):
        Ab = make_acts(synth.tensor_id(87, fmt, 4, M), M, K)
        A = bf16_dev(Ab)
        ref, _ = oracle.gemm(fmt, Ab, c, s, G, N)
        rg, _ = oracle.gemm(fmt, Ab, g[0], g[1], g[2], I)
        ru, _ = oracle.gemm(fmt, Ab, u[0], u[1], u[2], I)
        rgu = np.concatenate([rg, ru], axis=1)
        for Wt, r, what in ((W, ref, "plain"), (Wf, rgu, "fused"), (Wp, rgu, "paired")):
            y = vt.w4a16_gemm(A, Wt, opts={"grid": 2})
            again = vt.w4a16_gemm(A, Wt, opts={"grid": 2})
            torch.cuda.synchronize()
            st = Wt.stats()
            assert st["grid"] == 2 and st["tile_epilogue"] == 1, st
            check_rows(y.float().cpu().numpy(), r, what=f"{what} fmt={fmt} M={M}")
            assert np.array_equal(bf16_host_bits(y), bf16_host_bits(again)), what
    # three tokens take the CTA-wide epilogue
    vt.w4a16_gemm(bf16_dev(make_acts(synth.tensor_id(87, fmt, 4, 3), 3, K)), W, opts={"grid": 2})
    torch.cuda.synchronize()
    assert W.stats()["tile_epilogue"] == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_greedy_head_on_a_weight_of_many_row_tiles(fmt):
    # 469 row tiles of 8 k tiles: the default launch shape (152 CTAs) gives each CTA more
    # than three tiles
    N, K = 60000, 512
    c, s, G = make_weight(fmt, synth.tensor_id(87, fmt, 5), N, K)
    W = vt.PackedWeight.from_codes(to_dev(c), to_dev(s), G, fmt, N, K)
    ws = W.new_workspace(2)
    for M in (1, 2):
        Ab = make_acts(synth.tensor_id(87, fmt, 6, M), M, K)
        A = bf16_dev(Ab)
        y = vt.w4a16_gemm(A, W, workspace=ws)
        assert W.stats()["tile_epilogue"] == 1 and W.stats()["stage_k_tiles"] == 8
        tok, val = vt.w4a16_gemm_greedy(A, W, workspace=ws)
        torch.cuda.synchronize()
        assert W.stats()["tile_epilogue"] == 1
        ref, _ = oracle.gemm(fmt, Ab, c, s, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"lm_head-like fmt={fmt} M={M}")
        own, f = _first_argmax(bf16_host_bits(y))
        tok = tok.cpu().numpy()
        assert np.array_equal(tok, own), (M, tok, own)
        assert np.array_equal(val.cpu().numpy(), f[np.arange(M), own])
        check_against_oracle(tok, Ab, c, s, G, fmt, N, what=f"greedy fmt={fmt} M={M}")
    assert vt.workspace_status(ws) == 0
