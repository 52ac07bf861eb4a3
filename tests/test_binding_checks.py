"""CPU: the Python binding refuses tensors that the kernels cannot safely be handed --
host tensors, outputs of the wrong shape, type or inner stride, workspaces that are not
plain bytes -- before any library call.  A weight object without a library handle stands in
for a packed weight: none of these calls gets as far as using it."""
import ctypes

import pytest
import torch

import fp4_weight_only_nvfp4_gb300 as vt

N, K, M = 64, 128, 4


@pytest.fixture()
def W():
    w = vt.PackedWeight(ctypes.c_void_p(0), torch.empty(0, dtype=torch.uint8, device="meta"),
                        vt.NVFP4, N, K)
    w.I, w.paired = N // 2, True
    return w


def _A(m=M, k=K):
    return torch.zeros((m, k), dtype=torch.bfloat16)


def test_host_tensors_are_refused(W):
    A = _A()
    for call in (lambda: vt.w4a16_gemm(A, W), lambda: vt.w4a4_gemm(A, W, 1.0),
                 lambda: vt.w4a16_gemm_silu_mul(A, W), lambda: vt.w4a16_gemm_greedy(A, W),
                 lambda: vt.w4a16_gemm_noalloc(A, W),
                 lambda: vt.w4a16_gemm_moe(A, W, torch.zeros((M, 2), dtype=torch.int32))):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    with pytest.raises(ValueError, match="CUDA"):
        vt.workspace_status(torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        vt.quantize_act(A, vt.NVFP4)


def test_operand_shapes_are_checked_first(W):
    with pytest.raises(ValueError, match=r"\[M, K\]"):
        vt.w4a16_gemm(_A(k=K + 16), W)                       # K mismatch
    with pytest.raises(ValueError, match=r"\[M, K\]"):
        vt.w4a16_gemm(_A(k=2 * K)[:, ::2], W)                # inner stride 2
    with pytest.raises(ValueError, match=r"\[M, K\]"):
        vt.w4a16_gemm(_A().float(), W)                       # not bf16
    with pytest.raises(ValueError, match="topk_ids"):
        vt.w4a16_gemm_moe(_A(), W, torch.zeros((M, 2), dtype=torch.int64))
    with pytest.raises(ValueError, match="topk_ids"):
        vt.w4a16_gemm_moe(_A(), W, torch.zeros((M + 1, 2), dtype=torch.int32))


def test_output_shape_type_and_stride():
    ok = torch.empty((M, N + 8), dtype=torch.bfloat16)[:, :N]  # any row stride is fine
    vt._check_out(ok, M, N)
    for bad in (torch.empty((M - 1, N), dtype=torch.bfloat16),
                torch.empty((M, N - 1), dtype=torch.bfloat16),
                torch.empty((M * N,), dtype=torch.bfloat16),
                torch.empty((M, N), dtype=torch.float16),
                torch.empty((M, 2 * N), dtype=torch.bfloat16)[:, ::2]):
        with pytest.raises(ValueError, match="out must be"):
            vt._check_out(bad, M, N)


def test_grouped_sources_are_checked():
    E = 3
    codes = torch.zeros((E, N, K // 2), dtype=torch.uint8)
    scales = torch.zeros((E, N, K // 16), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        vt.PackedWeight.grouped(codes, scales, [1.0] * E, vt.NVFP4, E, N, K)
    with pytest.raises(ValueError, match=r"\[E, N, K/2\]"):
        vt.PackedWeight.grouped(codes[:2], scales[:2], [1.0] * E, vt.NVFP4, E, N, K)
    with pytest.raises(TypeError):
        vt.PackedWeight.grouped(codes.to(torch.int8), scales, [1.0] * E, vt.NVFP4, E, N, K)


def test_public_names():
    for name in vt.__all__:
        assert hasattr(vt, name), name
    for name in ("w4a16_gemm_moe", "w4a16_gemm_greedy", "w4a16_gemm_silu_mul", "w4a4_gemm",
                 "quantize_act"):
        assert name in vt.__all__
