"""GPU: the greedy head (vt_fp4_w4a16_gemm_greedy) -- per token the index of the largest
bf16 output, ties to the lowest index, without writing the outputs.

Checks: the index and value equal the first-occurrence argmax of the library's own bf16
output for the same inputs and launch shape (bit-exact: same sums); against the oracle the
index is a valid argmax within the GEMM tolerance, and equal to the oracle's choice when the
oracle's top value leads by more than twice that tolerance; ties across CTAs resolve to the
lowest index; the workspace's keys reset between calls."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import TOL, bf16_dev, bf16_host_bits, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _first_argmax(y_bits: np.ndarray):
    f = oracle.bf16_to_f32(y_bits)
    return np.argmax(f, axis=1).astype(np.int32), f


def check_against_oracle(tok: np.ndarray, Ab, codes, scales, G, fmt, N, what=""):
    ref, ref_bf = oracle.gemm(fmt, Ab, codes, scales, G, N)
    o_idx, _ = oracle.greedy(ref_bf)
    for m in range(ref.shape[0]):
        row = ref[m].astype(np.float64)
        top = row.max()
        tol = TOL * np.abs(row).max()
        assert row[tok[m]] >= top - tol, (what, m, tok[m], row[tok[m]], top)
        second = np.partition(row, -2)[-2] if row.size > 1 else -np.inf
        if top - second > 2 * tol:
            assert tok[m] == o_idx[m], (what, m, tok[m], o_idx[m])


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", [(1000, 1024), (5000, 512), (300, 2048)])
def test_greedy_matches_own_output_and_oracle(fmt, N, K):
    codes, scales, G = make_weight(fmt, synth.tensor_id(85, fmt, 1, N), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    ws = W.new_workspace(16)
    for M in (1, 3, 8, 16):
        Ab = make_acts(synth.tensor_id(85, fmt, 2, M * 100 + N), M, K)
        A = bf16_dev(Ab)
        y = vt.w4a16_gemm(A, W, workspace=ws)
        tok, val = vt.w4a16_gemm_greedy(A, W, workspace=ws)
        torch.cuda.synchronize()
        ybits = bf16_host_bits(y)
        own, f = _first_argmax(ybits)
        tok = tok.cpu().numpy()
        val = val.cpu().numpy()
        assert np.array_equal(tok, own), (M, tok, own)
        assert np.array_equal(val, f[np.arange(M), own])
        check_against_oracle(tok, Ab, codes, scales, G, fmt, N, what=f"fmt={fmt} M={M} N={N}")
    assert vt.workspace_status(ws) == 0


def test_greedy_ties_resolve_to_the_lowest_index_across_ctas():
    """Every row identical -> every output of a token equal -> index 0; then all rows zero
    except two identical rows far apart -> the lower of the two."""
    fmt, N, K = vt.NVFP4, 6000, 512
    c1, s1, G = make_weight(fmt, synth.tensor_id(86, 0, 1), 1, K)
    codes = np.repeat(c1, N, axis=0)
    scales = np.repeat(s1, N, axis=0)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    Ab = make_acts(synth.tensor_id(86, 0, 2), 5, K)
    tok, _ = vt.w4a16_gemm_greedy(bf16_dev(Ab), W)
    assert tok.cpu().numpy().tolist() == [0] * 5
    zc = np.zeros_like(codes)
    zc[700] = c1[0]
    zc[4100] = c1[0]
    W2 = vt.PackedWeight.from_codes(to_dev(zc), to_dev(scales), G, fmt, N, K)
    # activations equal to the dequantised row make both dot products positive and equal
    w = oracle.dequant(fmt, c1, s1, G, 1, K)[0]
    Ab2 = np.tile(torch.tensor(w, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
                  .view(np.uint16), (3, 1))
    tok2, val2 = vt.w4a16_gemm_greedy(bf16_dev(Ab2), W2)
    assert tok2.cpu().numpy().tolist() == [700] * 3
    assert np.all(val2.cpu().numpy() > 0)


def test_greedy_keys_reset_between_calls():
    fmt, N, K = vt.MXFP4, 2048, 1024
    codes, scales, G = make_weight(fmt, synth.tensor_id(87, 0, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    ws = W.new_workspace(8)
    for rep in range(4):
        M = (rep * 3) % 8 + 1
        Ab = make_acts(synth.tensor_id(87, 0, 2, rep), M, K)
        A = bf16_dev(Ab)
        tok, _ = vt.w4a16_gemm_greedy(A, W, workspace=ws)
        y = vt.w4a16_gemm(A, W, workspace=ws)
        torch.cuda.synchronize()
        own, _ = _first_argmax(bf16_host_bits(y))
        assert np.array_equal(tok.cpu().numpy(), own), rep
    head = ws[:256].cpu().numpy()
    assert not head[64:64 + 16 * 8 + 4].any()  # keys and counter are back to zero


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_greedy_many_tiles_per_cta_three_to_sixteen_tokens(fmt):
    # 469 row tiles of 32 k tiles: the default launch gives each CTA about three tiles, some
    # shared with a neighbour, so the 8-token tile carries each thread's best keys across
    # tiles (complete and reduced) before folding them; 16 tokens fold per tile.  Up to 8
    # tokens such a call (more than 4096 activation elements) takes the activation pre-pass
    # and stages of 16 k tiles
    N, K = 60000, 2048
    codes, scales, G = make_weight(fmt, synth.tensor_id(88, fmt, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    ws = W.new_workspace(16)
    for M in (3, 5, 8, 16):
        Ab = make_acts(synth.tensor_id(88, fmt, 2, M), M, K)
        A = bf16_dev(Ab)
        y = vt.w4a16_gemm(A, W, workspace=ws)
        torch.cuda.synchronize()
        st = W.stats()
        assert st["stage_k_tiles"] == (16 if M <= 8 else 8) and st["launches"] == 2, (M, st)
        tok, val = vt.w4a16_gemm_greedy(A, W, workspace=ws)
        torch.cuda.synchronize()
        st = W.stats()
        assert st["tile_epilogue"] == 0 and st["items"] >= 3 * (K // 64) * st["grid"], st  # >= 3 tiles per CTA
        assert st["stage_k_tiles"] == (16 if M <= 8 else 8), (M, st)
        own, f = _first_argmax(bf16_host_bits(y))
        tok = tok.cpu().numpy()
        assert np.array_equal(tok, own), (M, tok, own)
        assert np.array_equal(val.cpu().numpy(), f[np.arange(M), own])
        check_against_oracle(tok, Ab, codes, scales, G, fmt, N, what=f"many tiles fmt={fmt} M={M}")
    assert vt.workspace_status(ws) == 0
