"""GPU: prepack/unpack/dequant are bit-exact against the oracle, and the GPU quantiser produces
the oracle quantiser's bytes.  All through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, to_dev

pytestmark = pytest.mark.gpu


def _pack_codes(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _same_floats(a: np.ndarray, b: np.ndarray) -> bool:
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


@pytest.mark.parametrize("G", [1.0, 0.012345678, 3.0e-5])
def test_nvfp4_dequant_every_code_and_scale_byte(G):
    N, K = 256, 64  # row r: all four groups use scale byte r; k -> code k % 16
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 16, axis=1)
    W = vt.PackedWeight.from_codes(to_dev(_pack_codes(codes)), to_dev(scales), G, vt.NVFP4, N, K)
    got = W.dequant().cpu().numpy()
    want = oracle.dequant(oracle.NVFP4, _pack_codes(codes), scales, G, N, K)
    assert _same_floats(got, want)


@pytest.mark.parametrize("e0", [0, 30, 60, 90, 120, 150, 180, 210, 225])
def test_mxfp4_dequant_every_code_and_scale_byte(e0):
    # 30 consecutive exponents: the weight keeps the kernels' f16 scale encoding (a wider span
    # keeps raw bytes; tests/test_gpu_mx_wide.py covers all 256 bytes in one tensor)
    N, K = 31, 64
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    eb = np.minimum(e0 + np.arange(N), 254).astype(np.uint8)
    eb[-1] = 0xFF  # one NaN row
    scales = np.repeat(eb[:, None], K // 32, axis=1)
    W = vt.PackedWeight.from_codes(to_dev(_pack_codes(codes)), to_dev(scales), 1.0, vt.MXFP4, N, K)
    got = W.dequant().cpu().numpy()
    want = oracle.dequant(oracle.MXFP4, _pack_codes(codes), scales, 1.0, N, K)
    assert _same_floats(got, want)


def test_mxfp4_scale_window_edge():
    # exponents 29 apart still take the f16 encoding; both stay exact
    N, K = 2, 32
    codes = np.full((N, K), 7, np.uint8)  # +6
    scales = np.array([[200], [171]], np.uint8)
    W = vt.PackedWeight.from_codes(to_dev(_pack_codes(codes)), to_dev(scales), 1.0, vt.MXFP4, N, K)
    got = W.dequant().cpu().numpy()
    assert np.all(got[0] == 6.0 * 2.0 ** 73) and np.all(got[1] == 6.0 * 2.0 ** 44)


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", [(300, 160), (128, 64), (1, 32), (2049, 1024)])
def test_prepack_unpack_round_trip(fmt, N, K):
    rng = np.random.default_rng(N + K + fmt)
    g = vt.GROUP[fmt]
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    if fmt == vt.NVFP4:
        scales = rng.integers(0, 256, size=(N, K // g), dtype=np.uint8)
        G = 0.5
    else:
        scales = rng.integers(0, 256, size=(N, K // g), dtype=np.uint8)  # every byte
        G = 1.0
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    c2, s2 = W.unpack()
    assert np.array_equal(c2.cpu().numpy(), codes)
    assert np.array_equal(s2.cpu().numpy(), scales)


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_gate_up_prepack_round_trip_and_dequant(fmt):
    I, K = 200, 128
    rng = np.random.default_rng(7 + fmt)
    g = vt.GROUP[fmt]
    parts = []
    for i in range(2):
        c = rng.integers(0, 256, size=(I, K // 2), dtype=np.uint8)
        lo, hi = (0x20, 0x50) if fmt == vt.NVFP4 else (110, 130)
        s = rng.integers(lo, hi, size=(I, K // g), dtype=np.uint8)
        parts.append((c, s, [0.25, 0.75][i] if fmt == vt.NVFP4 else 1.0))
    W = vt.PackedWeight.gate_up(*[(to_dev(c), to_dev(s), G) for c, s, G in parts], fmt, I, K)
    c2, s2 = W.unpack()
    assert np.array_equal(c2.cpu().numpy(), np.concatenate([parts[0][0], parts[1][0]]))
    assert np.array_equal(s2.cpu().numpy(), np.concatenate([parts[0][1], parts[1][1]]))
    got = W.dequant().cpu().numpy()
    want = np.concatenate([oracle.dequant(fmt, c, s, G, I, K) for c, s, G in parts])
    assert _same_floats(got, want)


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("N,K", [(257, 512), (64, 4096)])
def test_gpu_quantizer_matches_oracle(fmt, N, K):
    Wb = synth.normal_bf16(0, synth.tensor_id(50, fmt, 1, N), 0.02, N, K)
    codes, scales, G = oracle.quantize(fmt, Wb)
    gc, gs, gg = vt.quantize(bf16_dev(Wb), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(gs.cpu().numpy(), scales)
    if fmt == vt.NVFP4:
        assert float(gg.item()) == G


def test_gpu_quantizer_ties_and_saturation():
    """Groups holding exact E2M1 midpoints (ties), values beyond the grid, zeros and a huge
    dynamic range: the GPU quantiser takes every rounding decision the oracle takes."""
    rng = np.random.default_rng(3)
    N, K = 64, 256
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75,
                     -2.5, -3.5, -5.0, 0.0])
    unit = 2.0 ** rng.integers(-20, 4, size=(N, K // 16))
    vals = np.tile(mids, (N, K // 16)) * np.repeat(unit, 16, axis=1)
    vals[:, 5::37] *= 1.7  # off-grid values
    Wb = torch.tensor(vals, dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    Wb = Wb.view(torch.int16).numpy().view(np.uint16)
    for fmt in (vt.NVFP4, vt.MXFP4):
        codes, scales, G = oracle.quantize(fmt, Wb)
        gc, gs, gg = vt.quantize(bf16_dev(Wb), fmt)
        torch.cuda.synchronize()
        assert np.array_equal(gc.cpu().numpy(), codes), fmt
        assert np.array_equal(gs.cpu().numpy(), scales), fmt
        if fmt == vt.NVFP4:
            assert float(gg.item()) == G
