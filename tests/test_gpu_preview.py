"""Preview variants of the routing (InfiniLM PR #604): top-4 preview routing
(Motivation), an expert budget on the block coreset (Summary; the pages name
the budget without defining it: here a cap on the experts a block keeps, the
first ones of the coreset order) and the probability-mass reading of the
coreset (Summary "block coreset routing", model card Usage "90% of its
routing": a slot's mass is its probability under the softmax over all
experts).  The CUDA path through the C ABI against the oracle on the same
seeded inputs: routing, probabilities, membership and weights bit for bit,
outputs on every row within the tolerance of parity_util."""
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


BUDGET_WORKLOADS = [W.BLOCK32, W.BLOCKS16_ZIPF, W.BY_NAME["rows2048-b8-tau0.9"],
                    W.BY_NAME["rows2048-b32-tau1"]]


@pytest.mark.parametrize("w", BUDGET_WORKLOADS, ids=lambda w: w.name)
def test_coreset_budget_bit_exact(w):
    case = Case(w)
    case.oracle_route()
    for B in (1, 16, 64):
        gpu = case.run(max_experts=B)
        assert_route_equal(gpu, case.ref)
        case.oracle_coreset(max_experts=B)
        assert_coreset_equal(gpu, case.ref)
        assert (gpu["core"] <= B).all()
    assert case.status["wait_timeout"] == 0


def test_forward_under_budget():
    """32-row block, budget 24 (below its ~120-expert coreset): outputs of every row."""
    case = Case(W.BLOCK32)
    gpu = case.run(max_experts=24)
    case.oracle_route()
    case.oracle_coreset(max_experts=24)
    assert_coreset_equal(gpu, case.ref)
    assert int(gpu["core"][0]) == 24
    y = case.oracle_forward()
    assert_close(gpu["y32"], y, what="y_f32")
    assert_close(gpu["y"], y, what="y")


def test_top4_preview_full_shape():
    """Top-4 preview routing at full shape (H 2048, 256 experts), coreset 0.9."""
    w = dataclasses.replace(W.BLOCK32, name="block32-top4", k=4)
    case = Case(w)
    gpu = case.run()
    case.oracle_route()
    assert_route_equal(gpu, case.ref)
    case.oracle_coreset()
    assert_coreset_equal(gpu, case.ref)
    y = case.oracle_forward()
    assert_close(gpu["y32"], y, what="y_f32")


def test_top4_preview_many_blocks():
    """Top-4 preview on 2048 rows in blocks of 16 (tensor-core router, large GEMMs)."""
    w = dataclasses.replace(W.BY_NAME["rows2048-b16-tau0.9"], name="rows2048-b16-top4", k=4)
    case = Case(w)
    gpu = case.run(max_experts=48)
    case.oracle_route()
    assert_route_equal(gpu, case.ref)
    case.oracle_coreset(max_experts=48)
    assert_coreset_equal(gpu, case.ref)
    y = case.oracle_forward()
    assert_close(gpu["y32"], y, what="y_f32")
    assert_close(gpu["y"], y, what="y")


def test_budget_rejects_negative():
    case = Case(W.TINY)
    idx, wt = case.layer.route(case.x, case.off)
    with pytest.raises(moe_block.MoeError):
        case.layer.coreset(case.off, idx, wt, 0.9, max_experts=-1)


PROB_WORKLOADS = [W.TINY, W.BLOCK32, W.BLOCKS16_ZIPF, W.BY_NAME["rows2048-b8-tau0.9"],
                  W.PREFILL8192]


@pytest.mark.parametrize("w", PROB_WORKLOADS, ids=lambda w: w.name)
def test_prob_mass_bit_exact(w):
    """moe_block_route_probs + moe_block_coreset_mass: ids, weights and the
    full-softmax probabilities bit for bit, the coreset under those masses bit for
    bit, and the outputs of every row within tolerance."""
    case = Case(w)
    gpu = case.run(probs=True)
    case.oracle_route(probs=True)
    assert_route_equal(gpu, case.ref)
    case.oracle_coreset(probs=True)
    assert_coreset_equal(gpu, case.ref)
    y = case.oracle_forward()
    assert_close(gpu["y32"], y, what="y_f32")
    assert_close(gpu["y"], y, what="y")
    assert case.status["wait_timeout"] == 0 and case.status["bad_expert_id"] == 0


def test_prob_mass_with_budget_and_same_ids():
    """The probability router gives the ids and weights of the plain router bit for
    bit; with a budget the coreset still follows the oracle."""
    case = Case(W.BLOCKS16_ZIPF)
    plain = {k: v.copy() for k, v in case.run().items()}
    gpu = case.run(probs=True, max_experts=12)
    assert np.array_equal(plain["idx"], gpu["idx"])
    assert np.array_equal(plain["w"].view(np.uint32), gpu["w"].view(np.uint32))
    case.oracle_route(probs=True)
    case.oracle_coreset(probs=True, max_experts=12)
    assert_coreset_equal(gpu, case.ref)
    assert (gpu["core"] <= 12).all()


def test_prob_mass_rejects_misaligned():
    """A mass pointer off the 4-byte grid is refused on the host (nothing launched)."""
    import ctypes
    case = Case(W.TINY)
    L = case.layer
    idx, wt, p = L.route(case.x, case.off, probs=True)
    lib = moe_block.load()
    rc = lib.moe_block_coreset_mass(
        L.plan.handle, case.R, ctypes.c_void_p(case.off.data_ptr()), 1,
        ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(wt.data_ptr()),
        ctypes.c_void_p(p.data_ptr() + 2), ctypes.c_float(0.9), 0,
        ctypes.c_void_p(L._keep.data_ptr()), ctypes.c_void_p(L._core.data_ptr()),
        ctypes.c_void_p(L._w_renorm.data_ptr()), None, ctypes.c_void_p(L.workspace.data_ptr()),
        L.workspace.numel(), None)
    assert rc == -1 and b"misaligned" in lib.moe_last_error()
