"""moe_block_route_noalloc: the router for callers that cannot allocate device memory.

Such callers (an engine that reserves all of its device memory up front, a
plugin that may only touch the buffers it is given) cannot provide a workspace;
this entry point keeps the router's scratch in a fixed 1 MiB array inside the
library.  These checks call it through the C ABI and compare it with
moe_block_route on the same inputs, bit for bit, on two calls in a row; the
second call runs on other rows with a logit bias, so leftovers of the first
call in the shared array would show.  The file is named so that pytest
collects it last.
"""
from __future__ import annotations

import pytest
import torch

from sparse_moe_layer_row_gb300 import moe_block, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    moe_block.load()
    w = W.BLOCK32
    T = W.make_tensors(w, device="cuda")
    layer = moe_block.MoeBlockLayer(T.w_router, T.w_gate, T.w_up, T.w_down, T.ws_gate, T.ws_up,
                                    T.ws_down, k=w.k, max_rows=1100, max_blocks=4)
    return w, T, layer


def _reference(layer, x, off, bias):
    idx, wt = layer.route(x, off, bias)
    torch.cuda.synchronize()
    return idx.clone(), wt.clone()


def test_noalloc_route_matches_workspace_route_on_two_calls(setup):
    w, T, layer = setup
    x2 = W.make_x(w, "cuda", rows=96, seed=77)
    off2 = torch.tensor([0, 40, 96], dtype=torch.int32, device="cuda")
    bias2 = torch.linspace(-1.0, 1.0, 2 * w.E, device="cuda").view(2, w.E).contiguous()
    calls = [(T.x, T.block_offsets, None), (x2, off2, bias2)]
    for x, off, bias in calls:
        ref_idx, ref_w = _reference(layer, x, off, bias)
        R = x.shape[0]
        idx = torch.full((R, w.k), -1, dtype=torch.int32, device="cuda")
        wt = torch.full((R, w.k), float("nan"), dtype=torch.float32, device="cuda")
        moe_block.moe_block_route_noalloc(layer.plan, x, off, bias, idx, wt)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(wt.view(torch.int32), ref_w.view(torch.int32))


def test_noalloc_route_rejects_calls_beyond_its_scratch(setup):
    w, T, layer = setup
    R = 1100  # 4 * 1100 * 256 bytes of logits > 1 MiB
    x = W.make_x(w, "cuda", rows=R, seed=3)
    off = torch.tensor([0, R], dtype=torch.int32, device="cuda")
    idx = torch.empty(R, w.k, dtype=torch.int32, device="cuda")
    wt = torch.empty(R, w.k, dtype=torch.float32, device="cuda")
    with pytest.raises(moe_block.MoeError) as ei:
        moe_block.moe_block_route_noalloc(layer.plan, x, off, None, idx, wt)
    assert ei.value.status == -2
    # the largest call that fits still runs and matches
    R = 1019
    x = x[:R].contiguous()
    off = torch.tensor([0, R], dtype=torch.int32, device="cuda")
    ref_idx, ref_w = _reference(layer, x, off, None)
    idx, wt = idx[:R], wt[:R]
    moe_block.moe_block_route_noalloc(layer.plan, x, off, None, idx, wt)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx) and torch.equal(wt, ref_w)


def test_noalloc_route_with_non_finite_logits_is_silent(setup):
    """A NaN and a -inf logit in one row (through the bias): the call still returns
    MOE_OK (the non-finite count stays inside the library's array and is not
    reported), that row ranks them last as moe_block_route does, and every row
    matches moe_block_route bit for bit."""
    w, T, layer = setup
    R = w.R
    bias = torch.zeros(1, w.E, dtype=torch.float32, device="cuda")
    bias[0, 7] = float("nan")
    bias[0, 11] = float("-inf")
    ref_idx, ref_w = _reference(layer, T.x, T.block_offsets, bias)
    idx = torch.full((R, w.k), -1, dtype=torch.int32, device="cuda")
    wt = torch.full((R, w.k), float("nan"), dtype=torch.float32, device="cuda")
    moe_block.moe_block_route_noalloc(layer.plan, T.x, T.block_offsets, bias, idx, wt)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx)
    assert torch.equal(wt.view(torch.int32), ref_w.view(torch.int32))
    assert not bool(((idx == 7) | (idx == 11)).any())
