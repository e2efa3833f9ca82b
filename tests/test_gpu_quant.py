"""Quantised expert weights (model card "Clover-35B-A3B-Preview -- CMF", Files:
the 8-bit and 4-bit expert files; the codec is this library's reading: blocks
of 32 weights along the input dimension with one bf16 scale, weight =
bf16(q * d)).  The streaming GEMMs read the codes and scales and dequantise
them in shared memory; the oracle dequantises the same codes in plain C and
runs its fp64 FFN.  Routing and coreset are bit-exact (the router stays
bf16), outputs within tolerance on every row, on the small path and on
larger calls (which stream quantised weights in 32-row units too)."""
from __future__ import annotations

import dataclasses

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


def _small(H=256, E=16, k=4, I=128, Is=128, rows=(32,), tau=0.9, seed=5):
    return W.Workload(name="quant", H=H, E=E, k=k, I=I, Is=Is, block_rows=tuple(rows), tau=tau,
                      sigma_r=0.05, x_seed=seed, w_seed=seed)


WORKLOADS = [W.TINY, W.BLOCK32, _small(rows=(5, 0, 7)), _small(H=512, I=64, Is=192, rows=(24, 8)),
             W.BY_NAME["rows2048-b32-tau0.9"]]


def _qcase(w, bits):
    T = W.make_tensors(w, device="cuda")
    return Case(w, T=T, quant=W.quantize_experts(T, bits))


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: f"{w.name}-{w.H}-{w.block_rows[:3]}")
def test_quantised_experts_match_the_oracle(w, bits):
    case = _qcase(w, bits)
    g = case.run()
    ref = case.oracle_route()
    assert_route_equal(g, ref)
    case.oracle_coreset()
    assert_coreset_equal(g, ref)
    case.oracle_forward()
    assert_close(g["y32"], ref["y"], what=f"y_f32 ({bits}-bit)")
    assert_close(g["y"], ref["y"], what=f"y ({bits}-bit)")
    st = case.status
    assert st["wait_timeout"] == 0 and st["bad_expert_id"] == 0 and st["nonfinite_output"] == 0


@pytest.mark.parametrize("bits", [8, 4])
def test_quantised_pass_equals_three_calls(bits):
    """moe_block_pass (fused front end) on a quantised layer gives the three calls'
    y bit for bit, and repeated calls are identical."""
    case = _qcase(W.BLOCK32, bits)
    ref = case.run()
    ys = []
    for _ in range(2):
        y = case.layer(case.x, case.off, W.BLOCK32.tau)
        torch.cuda.synchronize()
        ys.append(y.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(ys[0], ref["y"]) and np.array_equal(ys[1], ref["y"])


def test_quantised_differs_from_bf16_but_not_by_much():
    """The quantised layer is a different layer (its weights are rounded): its y is
    not the bf16 layer's, but close to it (8-bit round-to-nearest)."""
    T = W.make_tensors(W.BLOCK32, device="cuda")
    yb = Case(W.BLOCK32, T=T).run()["y32"]
    yq = Case(W.BLOCK32, T=T, quant=W.quantize_experts(T, 8)).run()["y32"]
    assert not np.array_equal(yb, yq)
    assert np.abs(yb - yq).max() < 0.05 * np.abs(yb).max()


def test_quantised_plan_rejects_bad_bits():
    T = W.make_tensors(W.TINY, device="cuda")
    Q = dataclasses.replace(W.quantize_experts(T, 8), bits=6)
    d = moe_block.moe_dims(256, 16, 4, 128, 128, 32, 1)
    with pytest.raises(ValueError):
        moe_block.Plan.quantized(d, T.w_router, Q)
    qw = moe_block.moe_quant_weights(6, *[getattr(Q, n).data_ptr() for n in moe_block._QFIELDS])
    import ctypes
    h = ctypes.c_void_p()
    rc = moe_block.load().moe_plan_create_quantized(ctypes.byref(d), ctypes.c_void_p(T.w_router.data_ptr()),
                                                    ctypes.byref(qw), ctypes.byref(h))
    assert rc == -2
