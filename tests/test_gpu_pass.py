"""moe_block_pass: one denoising pass (route -> coreset -> forward) in one call,
the kernels enqueued back to back.  Every output must equal the three separate
calls bit for bit, on every path, and match the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from tests.parity_util import Case, assert_close, assert_coreset_equal, assert_route_equal, bits32
from sparse_moe_layer_row_gb300 import moe_block, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    moe_block.load()


def _small(H=256, E=16, k=4, I=128, Is=128, rows=(32,), tau=0.9, seed=5):
    return W.Workload(name="pass", H=H, E=E, k=k, I=I, Is=Is, block_rows=tuple(rows), tau=tau,
                      sigma_r=0.05, x_seed=seed, w_seed=seed)


def run_pass(case: Case, tau=None, max_experts=0, probs=False, graph=False):
    tau = case.w.tau if tau is None else tau
    L, R, nb, w = case.layer, case.R, case.nb, case.w
    dev = case.dev
    out = dict(idx=torch.full((R, w.k), -1, dtype=torch.int32, device=dev),
               w=torch.full((R, w.k), float("nan"), device=dev),
               p=torch.full((R, w.k), float("nan"), device=dev) if probs else None,
               keep=torch.full((nb, (w.E + 31) // 32), -1, dtype=torch.int32, device=dev),
               core=torch.full((nb,), -1, dtype=torch.int32, device=dev),
               wr=torch.full((R, w.k), float("nan"), device=dev),
               empty=torch.full((nb,), -1, dtype=torch.int32, device=dev),
               y=torch.zeros(R, w.H, dtype=torch.bfloat16, device=dev),
               y32=torch.zeros(R, w.H, device=dev))

    def call():
        moe_block.moe_block_pass(L.plan, case.x, case.off, case.bias, tau, max_experts, out["idx"],
                                 out["w"], out["p"], out["keep"], out["core"], out["wr"],
                                 out["empty"], out["y"], out["y32"], L.workspace)
    if graph:
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            call()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            call()
        for t in out.values():
            if t is not None:
                t.zero_()
        g.replay()
    else:
        call()
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy().copy() for k, v in out.items() if v is not None and k != "y"}
    res["keep"] = bits32(res["keep"]).copy()
    res["y"] = out["y"].float().cpu().numpy().astype(np.float64)   # bf16 -> exact in fp64
    res["y32"] = res["y32"].astype(np.float64)
    return res


def _equal_to_calls(case: Case, tau=None, max_experts=0, probs=False):
    calls = {k: v.copy() for k, v in case.run(tau, max_experts=max_experts, probs=probs).items()}
    moe_block.moe_clear_device_status(case.layer.workspace)
    got = run_pass(case, tau, max_experts, probs)
    for key in calls:
        a, b = np.ascontiguousarray(calls[key]), np.ascontiguousarray(got[key])
        assert a.shape == b.shape and a.tobytes() == b.tobytes(), key   # bit for bit
    st = case.layer.status()
    assert st["wait_timeout"] == 0 and st["bad_expert_id"] == 0
    return got


SMALL = [W.TINY, W.BLOCK32, _small(rows=(5, 0, 7)), _small(rows=(13, 1, 1, 17)),
         _small(E=1024, k=8, I=64, Is=64, rows=(32,)), _small(E=64, k=32, rows=(20, 12)),
         _small(rows=(1,))]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"{w.name}-{w.E}-{w.k}-{w.block_rows}")
def test_small_pass_equals_three_calls(w):
    case = Case(w)
    got = _equal_to_calls(case)
    ref = case.oracle_route()
    assert_route_equal(got, ref)
    case.oracle_coreset()
    assert_coreset_equal(got, ref)
    case.oracle_forward()
    assert_close(got["y32"], ref["y"], what="y_f32 (pass)")
    assert_close(got["y"], ref["y"], what="y (pass)")


@pytest.mark.parametrize("tau", [0.5, 1.0])
def test_pass_tau_and_budget(tau):
    case = Case(W.BLOCK32)
    _equal_to_calls(case, tau=tau)
    _equal_to_calls(case, tau=tau, max_experts=20)


def test_pass_probability_mass():
    case = Case(W.BLOCK32)
    got = _equal_to_calls(case, probs=True)
    ref = case.oracle_route(probs=True)
    assert_route_equal(got, ref)
    case.oracle_coreset(probs=True)
    assert_coreset_equal(got, ref)


@pytest.mark.parametrize("w", [W.BLOCKS16_ZIPF, W.BY_NAME["rows2048-b8-tau0.9"]],
                         ids=lambda w: w.name)
def test_large_pass_equals_three_calls(w):
    _equal_to_calls(Case(w))


def test_pass_repeats_and_replays_bit_identically():
    """Repeated passes and a CUDA-graph replay give the same bits (the router's
    tickets are cleared by the call itself)."""
    case = Case(W.BLOCK32)
    a = run_pass(case)
    b = run_pass(case)
    c = run_pass(case, graph=True)
    for key in a:
        assert a[key].tobytes() == b[key].tobytes(), key
        assert a[key].tobytes() == c[key].tobytes(), key


def test_pass_on_a_workspace_full_of_garbage():
    """The call does not rely on the workspace's previous contents."""
    case = Case(W.BLOCK32)
    a = run_pass(case)
    case.layer.workspace.fill_(0xA5)
    moe_block.moe_clear_device_status(case.layer.workspace)
    b = run_pass(case)
    for key in a:
        assert a[key].tobytes() == b[key].tobytes(), key


def test_layer_call_is_the_pass():
    """MoeBlockLayer.__call__ runs moe_block_pass: its y equals the three calls'."""
    case = Case(W.BLOCK32)
    ref = case.run()
    y = case.layer(case.x, case.off, W.BLOCK32.tau)
    torch.cuda.synchronize()
    assert np.array_equal(y.float().cpu().numpy().astype(np.float64), ref["y"])


def test_pass_rejects_bad_arguments():
    case = Case(W.TINY)
    L = case.layer
    R, k = case.R, W.TINY.k
    args = [torch.empty(R, k, dtype=torch.int32, device="cuda"), torch.empty(R, k, device="cuda"),
            None, L._keep[:1], L._core[:1], L._w_renorm[:R], None,
            torch.empty(R, W.TINY.H, dtype=torch.bfloat16, device="cuda"), None, L.workspace]
    with pytest.raises(moe_block.MoeError):
        moe_block.moe_block_pass(L.plan, case.x, case.off, None, 0.0, 0, *args)
    with pytest.raises(moe_block.MoeError):
        moe_block.moe_block_pass(L.plan, case.x, case.off, None, 0.9, -1, *args)
