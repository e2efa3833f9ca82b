"""Preview variants of the routing (InfiniLM PR #604): top-4 preview routing
(Motivation) and an expert budget on the block coreset (Summary; the pages name
the budget without defining it: here a cap on the experts a block keeps, the
first ones of the coreset order).  The CUDA path through the C ABI against the
oracle on the same seeded inputs: routing, membership and weights bit for bit,
outputs within the tolerance of parity_util."""
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
    rows = list(range(0, w.R, 97))
    y = case.oracle_forward(rows=rows)
    assert_close(gpu["y32"], y, rows=rows, what="y_f32")


def test_budget_rejects_negative():
    case = Case(W.TINY)
    idx, wt = case.layer.route(case.x, case.off)
    with pytest.raises(moe_block.MoeError):
        case.layer.coreset(case.off, idx, wt, 0.9, max_experts=-1)
