"""CUDA path vs the CPU oracle, through the C ABI, on seeded synthetic inputs.

Routing ids and weights, coreset membership and renormalised weights are
compared bit for bit; layer outputs within |d| <= 2e-3 + 1e-2 |ref|.
Every workload, full-size ones included, compares routing, coreset and the
layer output on every row.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from sparse_moe_layer_row_gb300 import moe_block, workloads as W
import oracle
from tests.parity_util import (ATOL, Case, assert_close, assert_coreset_equal,
                               assert_route_equal, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_block.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _full(case: Case, tau=None):
    g = case.run(tau)
    ref = case.oracle_route()
    assert_route_equal(g, ref)
    case.oracle_coreset(tau)
    assert_coreset_equal(g, ref)
    case.oracle_forward()
    err = assert_close(g["y32"], ref["y"], what="y_f32")
    assert_close(g["y"], ref["y"], what="y (bf16)")
    assert case.status["wait_timeout"] == 0 and case.status["bad_expert_id"] == 0
    return err


def test_tiny_config():
    case = Case(W.TINY)
    _full(case)


def test_tiny_config_coreset_disabled():
    case = Case(W.TINY)
    _full(case, tau=1.0)
    assert case.gpu["core"][0] == len(set(case.gpu["idx"].reshape(-1).tolist()))


@pytest.mark.parametrize("tau", [0.9, 0.5, 0.99, 1.0])
def test_block32_full_shape(tau):
    case = Case(W.BLOCK32)
    _full(case, tau=tau)


def test_blocks16_zipf_bias():
    case = Case(W.BLOCKS16_ZIPF)
    _full(case)
    sizes = case.gpu["core"]
    assert sizes.min() < sizes.max(), "Zipf bias should make coreset sizes vary across blocks"


@pytest.mark.parametrize("w", W.ROWS2048, ids=lambda w: w.name)
def test_rows2048(w):
    case = Case(w)
    _full(case)


def test_prefill8192():
    case = Case(W.PREFILL8192)
    _full(case)


# --------------------------------------------------------------------------- edge cases

@pytest.mark.parametrize("base", [W.TINY, W.BLOCK32, W.BY_NAME["rows2048-b32-tau0.9"]],
                         ids=lambda w: w.name)
def test_outputs_beyond_fp16_range(base):
    """The down projections (routed and shared) times an exact power of two 2^s,
    chosen so that the expert outputs reach past fp16's largest value 65504 (at
    least four times).  Routing and h are unchanged and the layer is linear in
    those weights, so y scales by exactly 2^s: the staged outputs keep a
    power-of-two exponent per 32 columns, and
      * y equals 2^s times the unscaled layer's y up to fp16's resolution;
      * every row matches the oracle of the scaled layer, the tolerance's
        absolute part scaled by the same 2^s (the unscaled comparison, exactly);
      * no output is non-finite.
    Small path, and the CTA-pair / 256-row kernels of the large path."""
    T = W.make_tensors(base, device="cuda")
    small = Case(base, T=T)
    gs = small.run()
    ys = {k: gs[k].copy() for k in ("y32", "idx", "keep", "wr")}
    s = int(np.ceil(np.log2(4 * 65504 / np.abs(ys["y32"]).max()))) + 1
    big_T = dataclasses.replace(T, w_down=(T.w_down.float() * 2.0 ** s).to(torch.bfloat16),
                                ws_down=(T.ws_down.float() * 2.0 ** s).to(torch.bfloat16))
    assert torch.equal(big_T.w_down.float(), T.w_down.float() * 2.0 ** s)  # exact in bf16
    big = Case(base, T=big_T)
    gb = big.run()
    assert np.array_equal(gb["idx"], ys["idx"]) and np.array_equal(gb["keep"], ys["keep"])
    assert np.abs(gb["y32"]).max() > 4 * 65504
    assert big.status["nonfinite_output"] == 0
    # exact scaling up to the staging's rounding (fp16: 11 significant bits)
    assert np.allclose(gb["y32"], ys["y32"] * 2.0 ** s, rtol=2.0 ** -10, atol=2.0 ** (s - 20))
    ref = big.oracle_route()
    assert_route_equal(gb, ref)
    big.oracle_coreset()
    assert_coreset_equal(gb, ref)
    big.oracle_forward()
    assert_close(gb["y32"], ref["y"], what="y_f32 (scaled)", atol=ATOL * 2.0 ** s)
    assert_close(gb["y"], ref["y"], what="y (scaled)", atol=ATOL * 2.0 ** s)


def _small(H=256, E=16, k=4, I=128, Is=128, rows=(32,), tau=0.9, seed=5, sigma_r=0.05):
    return W.Workload(name="edge", H=H, E=E, k=k, I=I, Is=Is, block_rows=tuple(rows), tau=tau,
                      sigma_r=sigma_r, x_seed=seed, w_seed=seed)


@pytest.mark.parametrize("rows", [(1,), (3,), (5, 0, 7), (13, 1, 1, 30), (37, 64, 50)],
                         ids=str)
def test_ragged_blocks_and_rows(rows):
    _full(Case(_small(rows=rows)))


@pytest.mark.parametrize("E,k", [(20, 1), (20, 20), (37, 5), (64, 8), (40, 32)])
def test_expert_counts(E, k):
    _full(Case(_small(E=E, k=k, rows=(16, 9))))


@pytest.mark.parametrize("H,I,Is", [(512, 64, 192), (768, 320, 64), (256, 576, 128)])
def test_hidden_and_intermediate_sizes(H, I, Is):
    _full(Case(_small(H=H, I=I, Is=Is, rows=(24, 8))))


@pytest.mark.parametrize("H,I,Is,rows", [(768, 320, 192, (300, 300)), (512, 64, 192, (300, 300)),
                                         (256, 576, 128, (200, 100))], ids=str)
def test_hidden_and_intermediate_sizes_large(H, I, Is, rows):
    """The many-row kernels at other sizes: intermediate tiles cut short by I or
    Is (rows past them read as zeros), three 256-column down tiles (H = 768),
    the shared expert's K wrapping at Is != I; 600 rows take the CTA-pair down
    GEMM, 300 rows the streaming one beside the CTA-pair gate/up GEMM."""
    _full(Case(_small(H=H, I=I, Is=Is, rows=rows, E=16, k=4)))


def test_many_rows_small_shape_multichunk():
    """More than 256 rows per expert: several row chunks per expert and per shared unit."""
    w = _small(E=4, k=2, rows=(200, 300, 100), H=256, I=128, Is=64)
    _full(Case(w))


def test_router_ties_go_to_lower_id():
    w = _small()
    T = W.make_tensors(w, device="cuda")
    T.w_router[9] = T.w_router[2]
    T.w_router[14] = T.w_router[2]
    _full(Case(w, T=T))


def test_nonfinite_logits_counted_and_ranked_last():
    w = _small()
    T = W.make_tensors(w, device="cuda")
    bias = torch.zeros(1, w.E, dtype=torch.float32, device="cuda")
    bias[0, 3] = float("nan")
    bias[0, 5] = float("-inf")
    case = Case(w, T=T, bias=bias)
    g = case.run()
    ref = case.oracle_route()
    assert_route_equal(g, ref)
    assert case.status["nonfinite_logits"] == ref["nonfinite"] == 2 * w.R
    assert not np.isin(g["idx"], [3, 5]).any()


def test_empty_rows_keep_shared_expert_only():
    """At a very low tau the coreset shrinks to the heaviest expert or two; rows that
    selected none of them keep only the shared expert."""
    w = _small(E=32, k=2, rows=(32,), tau=0.05)
    case = Case(w)
    g = case.run()
    ref = case.oracle_route()
    assert_route_equal(g, ref)
    case.oracle_coreset()
    assert_coreset_equal(g, ref)
    assert int(ref["empty"].sum()) > 0
    case.oracle_forward()
    assert_close(g["y32"], ref["y"])
    assert case.status["empty_rows"] == int(ref["empty"].sum())


def test_bad_expert_ids_are_counted_not_fatal():
    w = _small()
    case = Case(w)
    L = case.layer
    idx, wt = L.route(case.x, case.off)
    keep, core, wr, empty = L.coreset(case.off, idx, wt, w.tau)
    idx2 = idx.clone()
    idx2[0, 0] = w.E + 5
    idx2[1, 1] = -2
    moe_block.moe_clear_device_status(L.workspace)
    L.coreset(case.off, idx2, wt, w.tau)
    y = L.forward(case.x, case.off, idx2, wr, keep)
    torch.cuda.synchronize()
    st = L.status()
    assert st["bad_expert_id"] == 2 and st["wait_timeout"] == 0
    assert torch.isfinite(y.float()).all()


def test_bad_block_offsets_are_counted():
    w = _small(rows=(16, 16))
    case = Case(w)
    bad = torch.tensor([0, 20, 12], dtype=torch.int32, device="cuda")
    idx, wt = case.layer.route(case.x, case.off)
    moe_block.moe_clear_device_status(case.layer.workspace)
    case.layer.coreset(bad, idx, wt, w.tau)
    torch.cuda.synchronize()
    assert case.layer.status()["bad_offsets"] == 1


def test_repeat_calls_are_deterministic_in_routing():
    case = Case(W.TINY)
    g1 = {k: v.copy() for k, v in case.run().items()}
    g2 = case.run()
    for key in ("idx", "w", "keep", "wr", "core"):
        assert np.array_equal(np.asarray(g1[key]), np.asarray(g2[key])), key
    assert np.allclose(g1["y32"], g2["y32"], rtol=1e-6, atol=1e-6)


def test_workspace_reuse_across_shapes():
    """One layer sized for the largest call serves smaller calls in between."""
    w = _small(rows=(64, 64))
    T = W.make_tensors(w, device="cuda")
    big = Case(w, T=T)
    _full(big)
    small_off = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    x5 = T.x[:5].contiguous()
    c2 = Case(w, T=T, block_offsets=[0, 5], x=x5)
    _full(c2)


# --------------------------------------------------------------------------- large-batch router

def _route_only(case: Case):
    L = case.layer
    idx, wt = L.route(case.x, case.off, case.bias)
    torch.cuda.synchronize()
    g = dict(idx=idx.cpu().numpy().copy(), w=wt.cpu().numpy().copy())
    ref = case.oracle_route()
    assert_route_equal(g, ref)
    return g, ref


@pytest.mark.parametrize("R,E,k,H", [(256, 256, 8, 256), (300, 48, 6, 512), (1000, 256, 16, 256),
                                     (513, 64, 1, 256), (257, 16, 4, 768)], ids=str)
def test_tensor_core_router_shapes(R, E, k, H):
    """Batches of >= 256 rows take the tensor-core screening path (E <= 256,
    E % 16 == 0, k <= 16); ids and weights stay bit-identical to the oracle."""
    w = _small(H=H, E=E, k=k, rows=(R,), sigma_r=0.02)
    _route_only(Case(w))


def test_tensor_core_router_ties_and_blocks():
    w = _small(E=64, k=8, rows=(100, 200, 84), sigma_r=0.02)
    T = W.make_tensors(w, device="cuda")
    T.w_router[40] = T.w_router[3]
    T.w_router[63] = T.w_router[3]
    bias = torch.randn(3, w.E, generator=torch.Generator().manual_seed(1)).to("cuda") * 0.1
    _route_only(Case(w, T=T, bias=bias))


def test_tensor_core_router_nonfinite_rows_fall_back():
    """NaN / -inf logits leave fewer comparable values; such rows are recomputed
    over every expert and still match the oracle."""
    w = _small(E=32, k=8, rows=(300,), sigma_r=0.02)
    T = W.make_tensors(w, device="cuda")
    bias = torch.zeros(1, w.E, dtype=torch.float32, device="cuda")
    bias[0, :20] = float("nan")
    bias[0, 20:26] = float("-inf")
    case = Case(w, T=T, bias=bias)
    g, ref = _route_only(case)
    assert (g["idx"][:, :6] >= 26).all()


def test_tensor_core_router_near_ties_around_the_bound():
    """Adversarial rows for the tensor-core screen (>= 256 rows): its approximate
    logits are within beta = H 2^-21 |x| |w| of the exact ones, and the exact top-k
    is recomputed over the experts within that bound of the k-th.  Here every row
    puts a twin pair of router rows at ranks k and k + 1: expert b is expert a
    with one element raised by one bf16 ulp, so their gap is x[h*] times that ulp,
    and x[h*] varies over the rows to sweep the gap from 1/100 of the row's beta to
    ten times it (both signs, so either twin wins).  Ids and weights stay bit-exact
    against the oracle on every row."""
    H, E, k, R = 256, 64, 8, 512
    g = torch.Generator().manual_seed(11)
    x0 = torch.randn(H, generator=g)
    hs = int(torch.argmax(x0.abs()))
    u = x0 / x0.norm()
    wr = torch.randn(E, H, generator=g) * 0.002
    for e in range(7):                       # ranks 1..7 for every row
        wr[e] = u * (0.06 + 0.01 * e) * 16
    a, b = 20, 41                            # the twins, ranks 8 and 9
    wr[a] = u * 0.04 * 16
    wr = wr.to(torch.bfloat16)
    wb = wr[a].clone()
    up = (wb[hs].view(torch.int16) + (1 if wb[hs] > 0 else -1)).view(torch.bfloat16)
    wb[hs] = up                              # one ulp away from zero
    wr[b] = wb
    delta = float(wr[b, hs].float() - wr[a, hs].float())
    # x[h*] per row: the gap x[h*] * delta against beta of the row
    xs = x0.repeat(R, 1)
    G = H * 2.0 ** -21
    wmax = float(wr.float().norm(dim=1).max()) * 1.001
    frac = torch.logspace(-2, 1, R // 2)
    targets = torch.cat([frac, -frac])
    for r in range(R):
        xn = float(x0.norm()) * 1.001
        xs[r, hs] = float(targets[r]) * G * xn * wmax / abs(delta)
    x = xs.to(torch.bfloat16)
    w = _small(H=H, E=E, k=k, rows=(R,), sigma_r=0.02)
    T = W.make_tensors(w, device="cuda")
    T.w_router.copy_(wr.to("cuda"))
    case = Case(w, T=T, x=x.to("cuda").contiguous())
    g_, ref = _route_only(case)
    # the construction did what it says: the twins hold ranks k and k + 1 and
    # their exact gaps straddle the screen's thresholds
    z = oracle.route(u16(x), u16(wr), [0, R], k, want_logits=True)[2]
    xn = np.linalg.norm(x.float().numpy(), axis=1) * 1.001
    gap = np.abs(z[:, a] - z[:, b]) / (G * xn * wmax)
    top = ref["idx"]
    on_edge = [(a in top[r]) != (b in top[r]) for r in range(R)]
    assert sum(on_edge) > 0.9 * R
    for lo, hi in ((0.01, 0.5), (0.5, 1.0), (1.0, 2.0), (2.0, 4.0)):
        assert ((gap > lo) & (gap < hi)).sum() >= 10, (lo, hi)


@pytest.mark.parametrize("rows", [(32,), (8,) * 80], ids=["one-block", "80-blocks"])
def test_largest_expert_count(rows):
    """E = 1024 (the largest supported), k = 8: the coreset's per-thread ranking
    (one block) and its sort over 1024 keys (80 blocks, >= 64), and the scatter's
    1024-column slot table."""
    w = _small(E=1024, k=8, rows=rows, H=256, I=64, Is=64)
    _full(Case(w))


def test_top32_of_64():
    """k = 32 (the largest supported) with 64 experts over 3 blocks."""
    _full(Case(_small(E=64, k=32, rows=(32, 17, 5))))
