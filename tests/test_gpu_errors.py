"""The device error path, exercised in forms that fault nothing (page "Tensor vs Expert vs Data
Parallelism for MoE Serving", section "Trade-offs, Gotchas, and What Goes Wrong": fixed buffers
fail loudly -- a failure must surface as an error the host reads, never as a hang):

* the CTA-pair GEMM launched without 2-CTA clusters: it either never starts (the runtime refuses
  the launch, reported as MOE_ERR_CUDA with the runtime's error name) or returns at once with
  device code 5;
* a wait that nothing completes runs out after a short wall-clock limit and records code 6.

After each, the context stays usable: the next forward pass is clean and matches the oracle.
"""
import time

import pytest

import mixture_experts_layer_83_b300 as moe
from moe_inputs.configs import SIGMOID, make_shape

from layer_check import full_check, gpu_forward
import moe_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SMALL = make_shape(T=96, d=256, E=16, k=4, F=128, Fs=64, dtype="bf16", score=SIGMOID,
                   bias_range=0.01, seed=103, name="after-error")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _layer_is_clean_and_correct():
    stats = full_check(SMALL, threads=4)
    res = gpu_forward(SMALL, moe_inputs.upload(SMALL, moe_inputs.host_inputs(SMALL)))
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(res["workspace"]) == (moe.MOE_OK, 0)
    return stats


def test_pair_gemm_without_clusters_never_runs_unpaired():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    rc = moe.moe_debug_unclustered_pair(ws, check=False)
    torch.cuda.synchronize()
    if rc == moe.MOE_OK:
        assert moe.moe_workspace_status(ws) == (moe.MOE_ERR_DEVICE, 5)
    else:
        assert rc == moe.MOE_ERR_CUDA
        print("launch refused:", moe.moe_last_cuda_error_name())
        assert moe.moe_last_cuda_error_name() != "cudaSuccess"
        assert moe.moe_workspace_status(ws) == (moe.MOE_OK, 0)
    print(_layer_is_clean_and_correct())


@pytest.mark.parametrize("limit_us", [20, 2000])
def test_wait_that_nothing_completes_runs_out_and_returns(limit_us):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_debug_wait_timeout(ws, limit_us * 1000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert moe.moe_workspace_status(ws) == (moe.MOE_ERR_DEVICE, 6)
    assert limit_us * 1e-6 <= elapsed < limit_us * 1e-6 + 2.0
    print(limit_us, elapsed, _layer_is_clean_and_correct())
