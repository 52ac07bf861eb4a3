"""GPU: the size limits.  The longest accepted K (110000, the largest multiple of the group
size not above it) on the decode path (M <= 16, the activation pre-pass: 1719 k tiles) and on
the tensor-core tile path (M > 16), against the oracle, with a ragged N; the next K up is
refused with VT_ERR_UNSUPPORTED on both paths instead of being computed."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu

K_MAX = {vt.NVFP4: 110000, vt.MXFP4: 109984}  # largest K <= 110000 that the group divides


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_longest_k_on_both_paths(fmt):
    N, K = 300, K_MAX[fmt]
    codes, scales, G = make_weight(fmt, synth.tensor_id(120, fmt, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    ws = W.new_workspace(40)
    for M, path in ((1, 1), (5, 1), (16, 1), (40, 2)):
        Ab = make_acts(synth.tensor_id(120, fmt, 2, M), M, K)
        y = vt.w4a16_gemm(bf16_dev(Ab), W, workspace=ws)
        torch.cuda.synchronize()
        assert W.stats()["path"] == path, (M, W.stats())
        ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
        check_rows(y.float().cpu().numpy(), ref, what=f"K={K} fmt={fmt} M={M}")
    assert vt.workspace_status(ws) == 0


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
def test_k_above_the_limit_is_refused(fmt):
    N, K = 128, 110016  # a multiple of both group sizes
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.full((N, K // (16 if fmt == vt.NVFP4 else 32)), 0x38 if fmt == vt.NVFP4 else 0x7F,
                     np.uint8)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), 1.0, fmt, N, K)
    ws = torch.zeros(32 << 20, dtype=torch.uint8, device="cuda")  # the K check comes first
    for M in (1, 40):
        A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(vt.VtError) as e:
            vt.w4a16_gemm(A, W, workspace=ws)
        assert e.value.status == _lib.VT_ERR_UNSUPPORTED and "110000" in str(e.value)
