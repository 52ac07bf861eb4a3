"""GPU: MXFP4 weights whose E8M0 scales span more exponents than the kernels' f16 scale
encoding holds (30 binades) -- every byte 0x00..0xFE is a finite scale 2^(e - 127) and 0xFF is
NaN, with no window ("native MXFP4 keep-quant + Qwen e2e", PR #38, commit "W2").  Such a weight
keeps its raw scale bytes in the packed tiles and the kernels apply each group's exact scale:
dequant and unpack are bit-exact over the whole byte range, and the GEMM on both paths matches
the oracle element by element, including output columns whose weights sit far below the
tensor's largest scale.

Element bound (besides the per-row tolerance of the other parity tests):
    |y_gpu - y_oracle| <= 2^-7 |y_oracle| + 2^-12 sum_k |A[m][k] w[n][k]|
the bf16 rounding of the output (2^-8 relative) with margin, plus the fp32 summation-order
difference of a K <= 1024 dot product (K 2^-24 sum |terms|, here with wide margin).  A column
whose weights were flushed to zero would fail it by its whole value."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, check_rows, make_acts, to_dev

pytestmark = pytest.mark.gpu


def _pack_codes(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _same_floats(a: np.ndarray, b: np.ndarray) -> bool:
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def _check_elems(y_gpu: np.ndarray, y_ref: np.ndarray, Ab: np.ndarray, wdeq: np.ndarray,
                 what: str = "") -> None:
    a = synth.bf16_bits_to_f32(Ab).astype(np.float64)
    mag = np.abs(a) @ np.abs(wdeq.astype(np.float64)).T
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bound = 2.0 ** -7 * np.abs(y_ref.astype(np.float64)) + 2.0 ** -12 * mag
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of bound, first at "
                           f"{np.argwhere(bad)[0]}: got {y_gpu[tuple(np.argwhere(bad)[0])]!r}, "
                           f"want {y_ref[tuple(np.argwhere(bad)[0])]!r}")


def _wide_weight(N: int, K: int, seed: int, lo: int = 20, hi: int = 230, per_row: bool = True):
    """Random codes; scale bytes spread over [lo, hi] (one exponent per row, or per group)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    if per_row:
        e = rng.integers(lo, hi + 1, size=(N, 1))
        scales = np.repeat(e, K // 32, axis=1).astype(np.uint8)
    else:
        scales = rng.integers(lo, hi + 1, size=(N, K // 32)).astype(np.uint8)
    scales[0, 0], scales[-1, -1] = lo, hi  # the span is exactly [lo, hi]
    return codes, scales


def test_mxfp4_dequant_every_code_and_scale_byte_in_one_tensor():
    N, K = 256, 64  # row r: both groups use scale byte r (0xFF: NaN); k -> code k % 16
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 32, axis=1)
    W = vt.PackedWeight.from_codes(to_dev(_pack_codes(codes)), to_dev(scales), 1.0, vt.MXFP4, N, K)
    got = W.dequant().cpu().numpy()
    want = oracle.dequant(oracle.MXFP4, _pack_codes(codes), scales, 1.0, N, K)
    assert _same_floats(got, want)
    c2, s2 = W.unpack()
    assert np.array_equal(c2.cpu().numpy(), _pack_codes(codes))
    assert np.array_equal(s2.cpu().numpy(), scales)


def test_mxfp4_scale_far_below_the_largest_is_exact():
    # an exponent 30 below the tensor's largest: no longer in the f16 window, kept exactly
    N, K = 2, 32
    codes = np.full((N, K), 7, np.uint8)  # +6
    scales = np.array([[200], [170]], np.uint8)
    W = vt.PackedWeight.from_codes(to_dev(_pack_codes(codes)), to_dev(scales), 1.0, vt.MXFP4, N, K)
    got = W.dequant().cpu().numpy()
    assert np.all(got[0] == 6.0 * 2.0 ** 73) and np.all(got[1] == 6.0 * 2.0 ** 43)


@pytest.mark.parametrize("N,K", [(300, 160), (1, 32), (2049, 1024)])
def test_mxfp4_unpack_round_trip_every_scale_byte(N, K):
    rng = np.random.default_rng(N * 3 + K)
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, size=(N, K // 32), dtype=np.uint8)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, vt.MXFP4, N, K)
    c2, s2 = W.unpack()
    assert np.array_equal(c2.cpu().numpy(), codes)
    assert np.array_equal(s2.cpu().numpy(), scales)
    got = W.dequant().cpu().numpy()
    assert _same_floats(got, oracle.dequant(oracle.MXFP4, codes, scales, 1.0, N, K))


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("N,K", [(300, 512), (1000, 1024)])
def test_wide_gemm_matches_oracle_both_paths(N, K, per_row):
    codes, scales = _wide_weight(N, K, seed=N + K + per_row, per_row=per_row)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, vt.MXFP4, N, K)
    wdeq = oracle.dequant(oracle.MXFP4, codes, scales, 1.0, N, K)
    ws = W.new_workspace(300)
    for M, force in ((1, 0), (2, 0), (5, 0), (8, 3), (13, 0), (16, 0), (40, 0), (300, 0), (7, 2)):
        Ab = make_acts(synth.tensor_id(70, N, M, K + per_row), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W, workspace=ws, opts={"force_path": force} if force else None)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(oracle.MXFP4, Ab, codes, scales, 1.0, N)
        got = y.float().cpu().numpy()
        what = f"N={N} K={K} M={M} force={force} per_row={per_row}"
        check_rows(got, ref, what=what)
        _check_elems(got, ref, Ab, wdeq, what=what)
    assert vt.workspace_status(ws) == 0


def test_wide_gemm_small_groups_alone():
    """Each row alternates two exponents 160 apart; odd tokens are zero on the large groups,
    so their outputs come from the small groups alone (about 2^-160 of the others)."""
    N, K = 260, 512
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 32), np.uint8)
    scales[:, 0::2], scales[:, 1::2] = 200, 40
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, vt.MXFP4, N, K)
    wdeq = oracle.dequant(oracle.MXFP4, codes, scales, 1.0, N, K)
    for M in (4, 12, 64):
        Ab = make_acts(synth.tensor_id(71, 0, M), M, K).copy()
        big = (np.arange(K) // 32) % 2 == 0
        Ab[1::2, big] = 0
        y = vt.w4a16_gemm(bf16_dev(Ab), W)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(oracle.MXFP4, Ab, codes, scales, 1.0, N)
        got = y.float().cpu().numpy()
        assert np.abs(ref[1::2]).max() < 2.0 ** -100 * np.abs(ref[0::2]).max()
        check_rows(got, ref, what=f"M={M}")
        _check_elems(got, ref, Ab, wdeq, what=f"M={M}")


def test_wide_gemm_subnormal_scales():
    """Scale bytes 0..3: weights 2^-128 .. 1.5 * 2^-124, fp32 subnormal or nearly so."""
    N, K = 200, 256
    codes, scales = _wide_weight(N, K, seed=11, lo=0, hi=60, per_row=True)
    scales[:50] = np.arange(50)[:, None] % 4
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, vt.MXFP4, N, K)
    wdeq = oracle.dequant(oracle.MXFP4, codes, scales, 1.0, N, K)
    for M in (3, 48):
        Ab = make_acts(synth.tensor_id(72, 0, M), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(oracle.MXFP4, Ab, codes, scales, 1.0, N)
        _check_elems(y.float().cpu().numpy(), ref, Ab, wdeq, what=f"M={M}")


def test_wide_gate_up_one_wide_half():
    """gate narrow (synthetic), up wide: the fused weight takes the exact path for both."""
    I, K = 640, 512
    Wb = synth.normal_bf16(0, synth.tensor_id(73, 0, 1), 0.02, I, K)
    gc, gs, _ = oracle.quantize(oracle.MXFP4, Wb)
    uc, us = _wide_weight(I, K, seed=7)
    W = vt.PackedWeight.gate_up((to_dev(gc), to_dev(gs), 1.0), (to_dev(uc), to_dev(us), 1.0),
                                vt.MXFP4, I, K)
    c2, s2 = W.unpack()
    assert np.array_equal(s2.cpu().numpy(), np.concatenate([gs, us]))
    codes, scales = np.concatenate([gc, uc]), np.concatenate([gs, us])
    wdeq = oracle.dequant(oracle.MXFP4, codes, scales, 1.0, 2 * I, K)
    for M in (1, 6, 16, 33):
        Ab = make_acts(synth.tensor_id(73, 0, 2, M), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(oracle.MXFP4, Ab, codes, scales, 1.0, 2 * I)
        _check_elems(y.float().cpu().numpy(), ref, Ab, wdeq, what=f"M={M}")


def test_wide_silu_mul_both_paths():
    I, K = 320, 256
    gc, gs = _wide_weight(I, K, seed=21, lo=100, hi=160)
    uc, us = _wide_weight(I, K, seed=22, lo=90, hi=170)
    W = vt.PackedWeight.gate_up((to_dev(gc), to_dev(gs), 1.0), (to_dev(uc), to_dev(us), 1.0),
                                vt.MXFP4, I, K, paired=True)
    for M in (3, 40):
        Ab = make_acts(synth.tensor_id(74, 0, M), M, K)
        y = vt.w4a16_gemm_silu_mul(bf16_dev(Ab), W)
        torch.cuda.synchronize()
        rg, _ = oracle.gemm(oracle.MXFP4, Ab, gc, gs, 1.0, I)
        ru, _ = oracle.gemm(oracle.MXFP4, Ab, uc, us, 1.0, I)
        ref = oracle.bf16_to_f32(oracle.silu_mul(np.concatenate([rg, ru], axis=1)))
        check_rows(y.float().cpu().numpy(), ref, what=f"silu M={M}")


def test_wide_w4a4_both_paths():
    N, K = 384, 512
    codes, scales = _wide_weight(N, K, seed=31, lo=60, hi=200)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, vt.MXFP4, N, K)
    for M in (2, 9, 40):
        Ab = make_acts(synth.tensor_id(75, 0, M), M, K)
        y = vt.w4a4_gemm(bf16_dev(Ab), W, 1.0)
        torch.cuda.synchronize()
        ref, _ = oracle.gemm_w4a4(oracle.MXFP4, Ab, 1.0, codes, scales, 1.0, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"w4a4 M={M}")


def test_wide_expert_in_a_grouped_weight():
    E, N, K, topk = 4, 256, 512, 2
    rng = np.random.default_rng(9)
    cs, ss = [], []
    for e in range(E):
        if e == 2:
            c, s = _wide_weight(N, K, seed=40 + e)
        else:
            c, s, _ = oracle.quantize(oracle.MXFP4,
                                      synth.normal_bf16(0, synth.tensor_id(76, e, 1), 0.02, N, K))
        cs.append(c)
        ss.append(s)
    W = vt.PackedWeight.grouped(to_dev(np.stack(cs)), to_dev(np.stack(ss)), [1.0] * E, vt.MXFP4,
                                E, N, K)
    for M in (3, 12):
        ids = np.stack([rng.permutation(E)[:topk] for _ in range(M)]).astype(np.int32)
        Ab = make_acts(synth.tensor_id(76, 9, M), M, K)
        y = vt.w4a16_gemm_moe(bf16_dev(Ab), W, to_dev(ids)).float().cpu().numpy()
        torch.cuda.synchronize()
        for m in range(M):
            for j in range(topk):
                e = int(ids[m, j])
                ref, _ = oracle.gemm(oracle.MXFP4, Ab[m:m + 1], cs[e], ss[e], 1.0, N)
                check_rows(y[m * topk + j:m * topk + j + 1], ref, what=f"moe m={m} e={e}")
