"""Failure path of the pipelined kernels (bounded waits), made to happen on
purpose without a fault: every wait of the GEMM and tensor-core router
pipelines gives up after a limit; a test-only limit of 1 ns makes them run
out.  The call must return (no CUDA error, the context usable), count the
timeouts in the device status word, and leave nothing behind: the next call
with the built-in limit, on the same workspace, gives the same outputs bit for
bit as before, and they match the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.parity_util import Case, assert_close, assert_coreset_equal, assert_route_equal
from sparse_moe_layer_row_gb300 import moe_block, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    moe_block.load()


def _abort_and_recover(case: Case):
    L = case.layer
    before = {k: v.copy() for k, v in case.run().items()}
    assert case.status["wait_timeout"] == 0
    L.plan.set_wait_limit(1)
    try:
        moe_block.moe_clear_device_status(L.workspace)
        case.run()
        torch.cuda.synchronize()
        st = L.status()
    finally:
        L.plan.set_wait_limit(0)
    assert st["wait_timeout"] > 0
    moe_block.moe_clear_device_status(L.workspace)
    after = case.run()
    assert case.status["wait_timeout"] == 0
    for key in ("idx", "w", "keep", "wr", "y32", "y"):
        assert np.array_equal(np.asarray(before[key]), np.asarray(after[key])), key
    ref = case.oracle_route()
    assert_route_equal(after, ref)
    case.oracle_coreset()
    assert_coreset_equal(after, ref)
    case.oracle_forward()
    assert_close(after["y32"], ref["y"], what="y_f32 after the aborted call")


def test_wait_limit_small_path():
    """32 rows: the streaming gate/up and down GEMMs (k_gemm) abort and drain."""
    _abort_and_recover(Case(W.TINY))


def test_wait_limit_large_path():
    """300 rows: the tensor-core router screen (k_route_tc), the CTA-pair gate/up
    GEMM and the streaming down GEMM (up to 512 rows) abort and drain."""
    w = W.Workload(name="abort-300", H=256, E=16, k=4, I=128, Is=128, block_rows=(300,),
                   tau=0.9, sigma_r=0.02, x_seed=9, w_seed=9)
    _abort_and_recover(Case(w))


def test_wait_limit_pair_down():
    """600 rows: the CTA-pair down GEMM (k_down_pair) aborts and drains too."""
    w = W.Workload(name="abort-600", H=256, E=16, k=4, I=128, Is=128, block_rows=(300, 300),
                   tau=0.9, sigma_r=0.02, x_seed=10, w_seed=9)
    _abort_and_recover(Case(w))


@pytest.mark.parametrize("bits", [8, 4])
def test_wait_limit_quantised(bits):
    """Quantised experts: the converter warps (voted waits, tensor-memory A
    slots) give up with the producer and the MMA thread, and the next call is
    unaffected (200 rows: a unit list of several rounds per CTA)."""
    w = W.Workload(name=f"abort-q{bits}", H=256, E=16, k=4, I=128, Is=128, block_rows=(100, 100),
                   tau=0.9, sigma_r=0.02, x_seed=11, w_seed=9)
    T = W.make_tensors(w, device="cuda")
    _abort_and_recover(Case(w, T=T, quant=W.quantize_experts(T, bits)))
