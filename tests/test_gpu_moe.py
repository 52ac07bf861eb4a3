"""GPU: the mixture-of-experts (grouped) decode GEMM.  Every output row (token m, slot j)
is a plain GEMM row of expert topk_ids[m, j], so the oracle is the plain oracle GEMM per
expert; the grouped prepack round-trips bit-exactly; results do not depend on the order of
the routing; an out-of-range expert id, or a pair beyond its expert's token tile, is
reported and skipped."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, bf16_host_bits, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _experts(fmt, E, N, K, tag):
    srcs = [make_weight(fmt, synth.tensor_id(89, tag, e, N), N, K) for e in range(E)]
    codes = to_dev(np.stack([s[0] for s in srcs]))
    scales = to_dev(np.stack([s[1] for s in srcs]))
    W = vt.PackedWeight.grouped(codes, scales, [s[2] for s in srcs], fmt, E, N, K)
    return srcs, W


def _routing(M, topk, E, seed, distinct=True):
    rng = np.random.default_rng(seed)
    if distinct:
        ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(M)])
    else:
        ids = rng.integers(0, E, size=(M, topk))
    return ids.astype(np.int32)


def _oracle(fmt, Ab, srcs, ids, N):
    M, topk = ids.shape
    ref = np.zeros((M * topk, N), np.float32)
    for e in np.unique(ids):
        rows = np.argwhere(ids == e)
        tok = rows[:, 0]
        c, s, G = srcs[e]
        y, _ = oracle.gemm(fmt, Ab[tok], c, s, G, N)
        for r, (m, j) in enumerate(rows):
            ref[m * topk + j] = y[r]
    return ref


def test_grouped_prepack_round_trip():
    fmt, E, N, K = vt.MXFP4, 5, 300, 512
    srcs, W = _experts(fmt, E, N, K, 1)
    codes, scales = W.unpack()
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), np.concatenate([s[0] for s in srcs]))
    assert np.array_equal(scales.cpu().numpy(), np.concatenate([s[1] for s in srcs]))


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("E,N,K", [(8, 256, 512), (33, 700, 1024)])
def test_moe_matches_oracle(fmt, E, N, K):
    srcs, W = _experts(fmt, E, N, K, 2 + fmt)
    ws = W.moe_workspace(16, 8)
    # one workspace for calls of every size, in both orders (no call's data may land on
    # another's split-K counters)
    for M, topk in ((1, 1), (1, 8), (5, 4), (16, 8), (5, 4), (16, 8), (2, 3)):
        ids = _routing(M, min(topk, E), E, seed=M * 10 + topk)
        Ab = make_acts(synth.tensor_id(89, fmt, synth.ROLE_A, M * 10 + topk), M, K)
        y = vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids), workspace=ws)
        torch.cuda.synchronize()
        check_rows(y.float().cpu().numpy(), _oracle(fmt, Ab, srcs, ids, N),
                   what=f"moe fmt={fmt} E={E} M={M} topk={topk}")
    assert vt.workspace_status(ws) == 0


def test_moe_shared_expert_and_order_independence():
    """All 16 tokens on expert 3 (one problem of 16 tokens) plus scattered slots; the same
    routing with each token's slots permuted gives the same rows, bit for bit."""
    fmt, E, N, K = vt.NVFP4, 12, 512, 1024
    srcs, W = _experts(fmt, E, N, K, 7)
    M, topk = 16, 4
    ids = _routing(M, topk, E, seed=99)
    ids[:, 0] = 3
    ids[:, 1:] = np.where(ids[:, 1:] == 3, 4, ids[:, 1:])
    Ab = make_acts(synth.tensor_id(89, 7, synth.ROLE_A), M, K)
    A = bf16_dev(Ab)
    y = vt.w4a16_gemm_moe(A, W, to_dev(ids))
    perm = ids[:, ::-1].copy()
    y2 = vt.w4a16_gemm_moe(A, W, to_dev(perm))
    torch.cuda.synchronize()
    check_rows(y.float().cpu().numpy(), _oracle(fmt, Ab, srcs, ids, N), what="shared expert")
    a = bf16_host_bits(y).reshape(M, topk, N)
    b = bf16_host_bits(y2).reshape(M, topk, N)[:, ::-1]
    assert np.array_equal(a, b)


def test_moe_out_of_range_expert_is_reported_and_skipped():
    fmt, E, N, K = vt.NVFP4, 4, 256, 512
    srcs, W = _experts(fmt, E, N, K, 8)
    ids = np.array([[0, 2], [9, 1]], np.int32)  # 9 is out of range
    Ab = make_acts(synth.tensor_id(89, 8, synth.ROLE_A), 2, K)
    ws = W.moe_workspace(2, 2)
    C = torch.full((4, N), 5.0, dtype=torch.bfloat16, device="cuda")
    vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids), out=C, workspace=ws)
    torch.cuda.synchronize()
    assert vt.workspace_status(ws) == 6
    got = C.float().cpu().numpy()
    assert np.all(got[2] == 5.0)  # the skipped pair's row is untouched
    ref = _oracle(fmt, Ab, srcs, np.array([[0, 2], [1, 1]], np.int32), N)
    check_rows(got[[0, 1, 3]], ref[[0, 1, 3]], what="valid pairs")


def test_moe_pairs_beyond_an_experts_token_tile_are_skipped():
    """Every token names expert 3 in both slots: with M = 5 (token tile of 8 rows) expert 3
    gets 10 pairs; the first 8 in pair order are computed, the last two (token 4) are
    skipped with status 6 and their rows left untouched."""
    fmt, E, N, K = vt.MXFP4, 4, 256, 512
    srcs, W = _experts(fmt, E, N, K, 9)
    M, topk = 5, 2
    ids = np.full((M, topk), 3, np.int32)
    Ab = make_acts(synth.tensor_id(89, 9, synth.ROLE_A), M, K)
    ws = W.moe_workspace(M, topk)
    C = torch.full((M * topk, N), 5.0, dtype=torch.bfloat16, device="cuda")
    vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids), out=C, workspace=ws)
    torch.cuda.synchronize()
    assert W.stats()["m_tile"] == 8
    assert vt.workspace_status(ws) == 6
    got = C.float().cpu().numpy()
    assert np.all(got[8:] == 5.0)
    ref = _oracle(fmt, Ab, srcs, ids, N)
    check_rows(got[:8], ref[:8], what="pairs within the token tile")


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_moe_both_grouped_modes_match_oracle(fmt):
    """Up to 8 tokens with K = 2048 (a 33 KB converted activation tile): the decode kernel
    groups the routing and converts the activations itself, one launch.  K = 8192 (129 KB)
    takes the pre-pass, two launches.  Token counts 1, 3 and 8, a token naming one expert
    twice, and every row against the oracle."""
    E, N = 6, 384
    for K, launches in ((2048, 1), (8192, 2)):
        srcs, W = _experts(fmt, E, N, K, 20 + fmt + K // 1024)
        ws = W.moe_workspace(8, 4)
        for M, topk in ((1, 4), (3, 2), (8, 4)):
            ids = _routing(M, topk, E, seed=M * 7 + K, distinct=(M != 3))
            if M == 3:
                ids[1] = [5, 5]
            Ab = make_acts(synth.tensor_id(89, 20 + fmt, K, M), M, K)
            y = vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids), workspace=ws)
            torch.cuda.synchronize()
            st = W.stats()
            assert st["m_tile"] == 8 and st["launches"] == launches, (K, M, st)
            tiles = min(M * topk, E) * 3  # 384 rows: three row tiles per expert
            if launches == 1 and tiles <= torch.cuda.get_device_properties(0).multi_processor_count:
                assert st["grid"] == tiles, (K, M, st)  # one whole row tile per CTA
            check_rows(y.float().cpu().numpy(), _oracle(fmt, Ab, srcs, ids, N),
                       what=f"moe fmt={fmt} K={K} M={M}")
        assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_moe_one_kernel_mode_ragged_k(fmt):
    """K = 544 (8.5 k tiles of 64): the in-kernel conversion of the one-launch mode zero-fills
    the last k tile past K, as the prepack zero-fills the weights there."""
    E, N, K = 5, 260, 544
    srcs, W = _experts(fmt, E, N, K, 30 + fmt)
    for M, topk in ((1, 3), (6, 2)):
        ids = _routing(M, topk, E, seed=M + 40)
        Ab = make_acts(synth.tensor_id(89, 30 + fmt, M), M, K)
        y = vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids))
        torch.cuda.synchronize()
        assert W.stats()["launches"] == 1
        check_rows(y.float().cpu().numpy(), _oracle(fmt, Ab, srcs, ids, N),
                   what=f"moe ragged K fmt={fmt} M={M}")


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_moe_long_one_kernel_call_uses_16_k_tile_stages(fmt):
    """16 experts of 3700 x 2048 (29 row tiles, the last ragged): 8 tokens that may name all 16
    experts give at least three row tiles per CTA, so the one-launch mode stages 16 k tiles at
    a time; one token naming 8 experts stays at 8.  Both against the oracle, row by row."""
    E, N, K = 16, 3700, 2048
    srcs, W = _experts(fmt, E, N, K, 50 + fmt)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, topk in ((8, 8), (8, 2), (1, 8)):
        ids = _routing(M, topk, E, seed=M * 13 + topk)
        Ab = make_acts(synth.tensor_id(89, 50 + fmt, M, topk), M, K)
        y = vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids))
        torch.cuda.synchronize()
        st = W.stats()
        long_call = min(M * topk, E) * 29 >= 3 * sms
        assert st["launches"] == 1 and st["stage_k_tiles"] == (16 if long_call else 8), (M, st)
        check_rows(y.float().cpu().numpy(), _oracle(fmt, Ab, srcs, ids, N),
                   what=f"moe long call fmt={fmt} M={M} topk={topk}")
