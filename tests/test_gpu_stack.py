"""Several MoE layers of a pass enqueued back to back and captured as one CUDA
graph (model card "Clover-35B-A3B-Preview -- CMF", Hardware: every pass as one
GPU submission).  Each layer's output in the stack equals the same layer called
alone, bit for bit, and that layer against the oracle; a replay of the captured
pass follows new inputs."""
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


def _layers(ws, Ts):
    return [moe_block.MoeBlockLayer(T.w_router, T.w_gate, T.w_up, T.w_down, T.ws_gate, T.ws_up,
                                    T.ws_down, k=w.k, max_rows=w.R, max_blocks=w.nb)
            for w, T in zip(ws, Ts)]


@pytest.mark.parametrize("rows", [(32,), (16, 16, 9, 23)], ids=["one-block", "four-blocks"])
def test_stack_layers_equal_single_calls(rows):
    base = dataclasses.replace(W.TINY, name="stack", block_rows=rows)
    ws = [dataclasses.replace(base, w_seed=100 + i, x_seed=10 + i) for i in range(3)]
    Ts = [W.make_tensors(w, device="cuda") for w in ws]
    off = Ts[0].block_offsets
    stack = moe_block.MoeStack(_layers(ws, Ts))
    outs = [o.clone() for o in stack([T.x for T in Ts], off, base.tau)]
    torch.cuda.synchronize()
    for i, (w, T) in enumerate(zip(ws, Ts)):
        case = Case(w, T=T, block_offsets=list(w.block_offsets()), bias=None)
        gpu = case.run()
        assert np.array_equal(outs[i].float().cpu().numpy().astype(np.float64), gpu["y"]), i
        assert_route_equal(gpu, case.oracle_route())
        assert_coreset_equal(gpu, case.oracle_coreset())
        assert_close(gpu["y"], case.oracle_forward(), what=f"layer {i} y")


def test_stack_graph_replay_is_one_submission():
    base = dataclasses.replace(W.TINY, name="stack")
    ws = [dataclasses.replace(base, w_seed=200 + i) for i in range(4)]
    Ts = [W.make_tensors(w, device="cuda") for w in ws]
    stack = moe_block.MoeStack(_layers(ws, Ts))
    x = Ts[0].x.clone()
    off = Ts[0].block_offsets
    eager = [o.clone() for o in stack(x, off, base.tau)]
    graph, outs = stack.capture(x, off, base.tau)
    for o in outs:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)
    # new input in the same buffer: the replayed pass follows it
    x.copy_(W.make_x(base, device="cuda", seed=base.x_seed + 1))
    graph.replay()
    torch.cuda.synchronize()
    replayed = [o.clone() for o in outs]
    assert not torch.equal(replayed[0], eager[0])
    again = stack(x, off, base.tau)
    torch.cuda.synchronize()
    for a, b in zip(replayed, again):
        assert torch.equal(a, b)
    # the graph's outputs are its own: eager calls of the layers leave them alone
    x.copy_(W.make_x(base, device="cuda", seed=base.x_seed + 2))
    stack(x, off, base.tau)
    torch.cuda.synchronize()
    for a, b in zip(outs, replayed):
        assert torch.equal(a, b)
