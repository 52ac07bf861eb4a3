"""GPU: the failure path of the kernels' bounded waits, without a GPU fault.

Every device-side wait of the decode and prefill kernels has a limit; a wait that runs out
sets VT_ERR_TIMEOUT in the workspace status word and the kernel finishes without waiting
any further.  The test makes the waits run out on purpose: the `withhold_weights` hook
stops the weight producer from issuing any copy (so nothing is in flight), and a 20 ms
limit keeps the test short.  It then checks that the status word reports the timeout, that
reading it clears it, and that the next call on the same workspace (its split-K counters
included) is correct."""
import time

import pytest
import torch

import oracle
import synth
import fp4_weight_only_nvfp4_gb300 as vt
from fp4_weight_only_nvfp4_gb300 import _lib
from gpu_helpers import bf16_dev, check_rows, make_acts, make_weight, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path,M", [(1, 1), (1, 12), (2, 40)])
def test_bounded_wait_times_out_and_the_workspace_recovers(path, M):
    fmt, N, K = vt.NVFP4, 640, 2048
    codes, scales, G = make_weight(fmt, synth.tensor_id(80, path, 1), N, K)
    W = vt.PackedWeight.from_codes(to_dev(codes), to_dev(scales), G, fmt, N, K)
    Ab = make_acts(synth.tensor_id(80, path, 2, M), M, K)
    A = bf16_dev(Ab)
    ws = W.new_workspace(M)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    vt.w4a16_gemm(A, W, workspace=ws,
                  opts={"force_path": path, "withhold_weights": 1, "wait_limit_us": 20000})
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert W.stats()["path"] == path
    assert elapsed < 1.5, elapsed  # each role gives up after its first 20 ms wait
    assert vt.workspace_status(ws) == _lib.VT_ERR_TIMEOUT
    assert vt.workspace_status(ws) == _lib.VT_OK  # reading cleared it
    y = vt.w4a16_gemm(A, W, workspace=ws, opts={"force_path": path})
    torch.cuda.synchronize()
    ref, _ = oracle.gemm(fmt, Ab, codes, scales, G, N)
    check_rows(y.float().cpu().numpy(), ref, what=f"after timeout path={path} M={M}")
    assert vt.workspace_status(ws) == _lib.VT_OK
