"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and
the CPU oracle on the same seeded inputs and compare.

Tolerance for floating-point outputs (bf16 inputs, fp32 accumulation):
|gpu - ref| <= ATOL + RTOL * |ref| elementwise, ref = the oracle's fp64 result.
Routing ids, router weights, coreset membership and renormalised weights are
compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_moe_layer_row_gb300 import moe_block, workloads as W

ATOL = 2e-3
RTOL = 1e-2

# worst element of each output comparison as a fraction of the tolerance,
# keyed by test and output (printed in the session summary, see conftest.py)
WORST: dict = {}


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a).view(np.uint32)


class Case:
    """One workload on the GPU: inputs, a layer with its workspace, and GPU results."""

    def __init__(self, w: W.Workload, device="cuda", T: W.Tensors | None = None,
                 block_offsets=None, bias=None, x=None, quant: W.QuantExperts | None = None):
        """``quant``: the experts quantised (workloads.quantize_experts of T); the GPU
        layer reads those codes and the oracle's FFN runs on the oracle's own
        dequantisation of them."""
        self.w = w
        self.quant = quant
        self.dev = torch.device(device)
        self.T = T if T is not None else W.make_tensors(w, device=self.dev)
        self.x = self.T.x if x is None else x
        self.off = (self.T.block_offsets if block_offsets is None
                    else torch.tensor(block_offsets, dtype=torch.int32, device=self.dev))
        self.bias = self.T.bias if bias is None else bias
        self.R = self.x.shape[0]
        self.nb = self.off.shape[0] - 1
        if quant is not None:
            self.layer = moe_block.MoeBlockLayer.quantized(
                self.T.w_router, quant, k=w.k, max_rows=max(self.R, 1), max_blocks=self.nb)
        else:
            self.layer = moe_block.MoeBlockLayer(
                self.T.w_router, self.T.w_gate, self.T.w_up, self.T.w_down, self.T.ws_gate,
                self.T.ws_up, self.T.ws_down, k=w.k, max_rows=max(self.R, 1), max_blocks=self.nb)
        moe_block.moe_clear_device_status(self.layer.workspace)

    def run(self, tau: float | None = None, max_experts: int = 0, probs: bool = False):
        """route -> coreset -> forward on the GPU.  ``probs``: the probability-mass
        reading (moe_block_route_probs, then moe_block_coreset_mass with topk_p)."""
        tau = self.w.tau if tau is None else tau
        L = self.layer
        p = None
        if probs:
            idx, wt, p = L.route(self.x, self.off, self.bias, probs=True)
        else:
            idx, wt = L.route(self.x, self.off, self.bias)
        keep, core, wr, empty = L.coreset(self.off, idx, wt, tau, max_experts=max_experts, mass=p)
        y32 = torch.empty(self.R, self.w.H, dtype=torch.float32, device=self.dev)
        y = L.forward(self.x, self.off, idx, wr, keep, y_f32=y32)
        torch.cuda.synchronize()
        self.gpu = dict(idx=idx.cpu().numpy().copy(), w=wt.cpu().numpy().copy(),
                        keep=bits32(keep).copy(), core=core.cpu().numpy().copy(),
                        wr=wr.cpu().numpy().copy(), empty=empty.cpu().numpy().copy(),
                        y=y.float().cpu().numpy().astype(np.float64),
                        y32=y32.cpu().numpy().astype(np.float64))
        if p is not None:
            self.gpu["p"] = p.cpu().numpy().copy()
        self.status = L.status()
        return self.gpu

    # ---- oracle side
    def oracle_route(self, nthreads=None, probs: bool = False):
        nthreads = nthreads or oracle.default_threads()
        off = self.off.cpu().numpy()
        bias = None if self.bias is None else self.bias.cpu().numpy()
        out = oracle.route(u16(self.x), u16(self.T.w_router), off, self.w.k, bias=bias,
                           nthreads=nthreads, want_probs=probs)
        idx, wt, z, nf = out[:4]
        self.ref = dict(idx=idx, w=wt, nonfinite=nf, off=off)
        if probs:
            self.ref["p"] = out[4]
        return self.ref

    def oracle_coreset(self, tau=None, max_experts: int = 0, probs: bool = False):
        tau = self.w.tau if tau is None else tau
        r = self.ref
        keep, core, wr, empty, bad = oracle.coreset(r["off"], r["idx"], r["w"], self.w.E, tau,
                                                    max_experts=max_experts,
                                                    mass=r["p"] if probs else None)
        r.update(keep=keep, core=core, wr=wr, empty=empty)
        return r

    def oracle_forward(self, rows=None, nthreads=None):
        nthreads = nthreads or oracle.default_threads()
        r = self.ref
        sel = rows if rows is not None else range(self.R)
        off = r["off"]
        mask = oracle.keep_mask(r["keep"], self.w.E)
        bor = np.searchsorted(off, np.arange(self.R), side="right") - 1
        used = set()
        for row in sel:
            for j in range(self.w.k):
                e = int(r["idx"][row, j])
                if mask[bor[row], e]:
                    used.add(e)
        if self.quant is not None:
            Q, b = self.quant, self.quant.bits

            def dq(codes, scale):
                return oracle.dequant(codes.detach().cpu().numpy(), u16(scale), b)
            def gud(e):   # the gate and up matrices of the interleaved layout
                gq, gd, uq, ud = Q.gate_and_up(e)
                return dq(gq, gd), dq(uq, ud)
            experts = {e: (*gud(e), dq(Q.down[e], Q.down_scale[e])) for e in sorted(used)}
            shared = (*gud(None), dq(Q.shared_down, Q.shared_down_scale))
        else:
            experts = {e: (u16(self.T.w_gate[e]), u16(self.T.w_up[e]), u16(self.T.w_down[e]))
                       for e in sorted(used)}
            shared = (u16(self.T.ws_gate), u16(self.T.ws_up), u16(self.T.ws_down))
        y = oracle.forward(u16(self.x), off, r["idx"], r["wr"], r["keep"], experts, shared,
                           self.w.E, rows=None if rows is None else list(rows),
                           nthreads=nthreads)
        r["y"] = y
        return y


def assert_route_equal(gpu, ref):
    assert np.array_equal(gpu["idx"], ref["idx"]), (
        f"top-k ids differ in {int((gpu['idx'] != ref['idx']).any(axis=1).sum())} rows")
    assert np.array_equal(bits32(gpu["w"]), bits32(ref["w"])), "router weights differ"
    if "p" in gpu or "p" in ref:
        assert np.array_equal(bits32(gpu["p"]), bits32(ref["p"])), "probability masses differ"


def assert_coreset_equal(gpu, ref):
    assert np.array_equal(gpu["core"], ref["core"]), "coreset sizes differ"
    assert np.array_equal(gpu["keep"], ref["keep"]), "coreset membership differs"
    assert np.array_equal(bits32(gpu["wr"]), bits32(ref["wr"])), "renormalised weights differ"
    assert np.array_equal(gpu["empty"], ref["empty"]), "empty-row counts differ"


def assert_close(got, ref, rows=None, what="y", atol=ATOL):
    """Elementwise |got - ref| <= atol + RTOL |ref| on every element (or on ``rows``).
    Records the worst element as a fraction of its tolerance under the running
    test's name; returns the largest absolute error."""
    import os
    if rows is not None:
        got, ref = got[list(rows)], ref[list(rows)]
    err = np.abs(got - ref)
    tol = atol + RTOL * np.abs(ref)
    bad = err > tol
    frac = float((err / tol).max()) if err.size else 0.0
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    key = f"{test} {what} ({got.shape[0]} rows)"
    WORST[key] = max(WORST.get(key, 0.0), frac)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max abs err {err.max():.3e}, worst {frac:.3f} of the tolerance")
    return float(err.max())
