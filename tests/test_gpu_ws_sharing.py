"""GPU: one workspace serving weights of different shapes, call after call without a host
synchronisation (eagerly and in a CUDA graph).  Each weight's activation and partial-sum
regions overlap the other's split-K counters, so every call must start from zeroed
counters; the outputs are checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


def _weights(fmt):
    # W1: 80 row tiles (counters over bytes 256..576 of the workspace), 32 k tiles, row
    # tiles shared by two CTAs; W2: 4 row tiles of 64 k tiles, whose activation scales
    # start at byte 512 and so overwrite W1's last counters.
    shapes = [(10240, 2048), (512, 4096)]
    out = []
    for i, (N, K) in enumerate(shapes):
        c, s, G = make_weight(fmt, synth.tensor_id(98, fmt, i), N, K)
        W = vt.PackedWeight.from_codes(to_dev(c), to_dev(s), G, fmt, N, K)
        out.append((W, c, s, G, N, K))
    return out


def _plan(ws_list):
    """(weight index, M) calls alternating between the shapes."""
    return [(0, 1), (1, 1), (0, 3), (1, 5), (0, 16), (1, 2), (0, 1), (1, 16), (0, 8)]


@pytest.mark.parametrize("fmt", [vt.NVFP4, vt.MXFP4])
@pytest.mark.parametrize("graph", [False, True])
def test_shared_workspace_across_shapes(fmt, graph):
    ws_list = _weights(fmt)
    plan = _plan(ws_list)
    wsz = max(W.workspace_bytes(16) for W, *_ in ws_list)
    ws = torch.zeros(wsz, dtype=torch.uint8, device="cuda")
    acts = [make_acts(synth.tensor_id(99, fmt, i, M), M, ws_list[wi][5]) for i, (wi, M) in enumerate(plan)]
    A = [bf16_dev(a) for a in acts]
    C = [torch.full((M, ws_list[wi][4]), 3.0, dtype=torch.bfloat16, device="cuda") for wi, M in plan]
    s = torch.cuda.Stream()

    def issue():
        for i, (wi, M) in enumerate(plan):
            vt.w4a16_gemm(A[i], ws_list[wi][0], out=C[i], workspace=ws, stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        issue()  # eager (also loads the kernels before any capture)
    s.synchronize()
    if graph:
        for c in C:
            c.fill_(3.0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            issue()
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
        s.synchronize()
    for i, (wi, M) in enumerate(plan):
        W, c, sc, G, N, K = ws_list[wi]
        ref, _ = oracle.gemm(fmt, acts[i], c, sc, G, N)
        check_rows(C[i].float().cpu().numpy(), ref, what=f"call {i} (weight {wi}, M={M})")
    assert vt.workspace_status(ws) == 0
