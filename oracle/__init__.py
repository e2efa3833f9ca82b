"""CPU oracle for the block-coreset sparse MoE FFN (ctypes wrapper of moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  It imports nothing
from the CUDA package; arrays come in as numpy (bf16 as uint16 bit patterns).

Each function follows the step of the method named in its docstring; the
readings of the pages that fix the arithmetic are listed at the top of
moe_oracle.c.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def use_library(path: str | None):
    """Swap in another build of moe_oracle.c (None: the default one).  Used by the
    mutation tests, which plant mistakes in a copy of the source."""
    global _lib
    _lib = None if path is None else _configure(ctypes.CDLL(path))


def _configure(L):
    if True:
        P = ctypes.c_void_p
        i = ctypes.c_int
        L.moe_oracle_exp_c.restype = ctypes.c_float
        L.moe_oracle_exp_c.argtypes = [ctypes.c_float]
        L.moe_oracle_logit.restype = ctypes.c_float
        L.moe_oracle_logit.argtypes = [P, P, i]
        L.moe_oracle_route.restype = ctypes.c_long
        L.moe_oracle_route.argtypes = [P, P, P, P, i, i, i, i, i, P, P, P, P, i]
        L.moe_oracle_coreset.restype = ctypes.c_long
        L.moe_oracle_coreset.argtypes = [P, i, i, i, i, P, P, P, ctypes.c_float, P, P, P, P, i]
        L.moe_oracle_expert_ffn.restype = None
        L.moe_oracle_expert_ffn.argtypes = [P, P, P, P, i, i, P]
        L.moe_oracle_dequant.restype = ctypes.c_int
        L.moe_oracle_dequant.argtypes = [P, P, i, i, i, P]
        L.moe_oracle_forward.restype = ctypes.c_int
        L.moe_oracle_forward.argtypes = [P, P, i, i, i, i, i, i, i, P, P, P, P, P, P, P, P, P,
                                         P, i]
    return L


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def exp_c(t: float) -> float:
    """Routing exponential on t <= 0 (Cody-Waite + degree-7 Taylor; reading 3)."""
    return float(lib().moe_oracle_exp_c(ctypes.c_float(t)))


def logit(x_row: np.ndarray, w_row: np.ndarray) -> float:
    """One router logit in the fixed lane/stripe summation order (reading 1)."""
    x_row, w_row = _u16(x_row), _u16(w_row)
    return float(lib().moe_oracle_logit(_ptr(x_row), _ptr(w_row), x_row.shape[0]))


def route(x, w_router, block_offsets, k, bias=None, want_logits=False, nthreads=1,
          want_probs=False):
    """Router logits -> top-k (z desc, id asc) -> softmax over the selected k.

    Model card "Clover-35B-A3B-Preview -- CMF", intro (256 experts, top-8).
    Returns (topk_idx int32 [R,k], topk_w fp32 [R,k], logits fp32 [R,E] or None,
    number of non-finite logits).  With ``want_probs`` a fifth value: topk_p fp32
    [R,k], the selected experts' probabilities under the full softmax over all E
    experts (reading 3b: the other mass reading of "90% of its routing",
    InfiniLM PR #604, Summary).
    """
    x, w_router = _u16(x), _u16(w_router)
    R, H = x.shape
    E = w_router.shape[0]
    off = np.ascontiguousarray(block_offsets, dtype=np.int32)
    nb = off.shape[0] - 1
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    idx = np.zeros((R, k), np.int32)
    w = np.zeros((R, k), np.float32)
    z = np.zeros((R, E), np.float32) if want_logits else None
    p = np.zeros((R, k), np.float32) if want_probs else None
    nf = lib().moe_oracle_route(_ptr(x), _ptr(w_router), _ptr(b), _ptr(off), nb, R, H, E, k,
                                _ptr(idx), _ptr(w), _ptr(p), _ptr(z), int(nthreads))
    if nf < 0:
        raise ValueError("oracle route: invalid arguments")
    if want_probs:
        return idx, w, z, int(nf), p
    return idx, w, z, int(nf)


def coreset(block_offsets, topk_idx, topk_w, E, tau, max_experts=0, mass=None):
    """Per-block coreset carrying >= tau of the block's routing mass, then renormalise.

    Model card "Clover-35B-A3B-Preview -- CMF", Usage (90% of the block's
    routing); InfiniLM PR #604, Summary (block coreset routing; expert budget).
    max_experts > 0 caps the coreset at that many experts: the first ones of
    the (mass desc, id asc) order (the pages name the budget only; this is the
    reading taken).  ``mass`` (fp32 [R,k], e.g. the topk_p of ``route``) gives
    the slots' masses; None takes them from topk_w.  The renormalised weights
    always come from topk_w.  Returns (keep uint32 [nb, ceil(E/32)], core_size
    int32 [nb], w_renorm fp32 [R,k], n_empty int32 [nb], n_bad_ids).
    """
    off = np.ascontiguousarray(block_offsets, dtype=np.int32)
    nb = off.shape[0] - 1
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    R, k = idx.shape
    words = (E + 31) // 32
    keep = np.zeros((nb, words), np.uint32)
    cs = np.zeros(nb, np.int32)
    wr = np.zeros((R, k), np.float32)
    ne = np.zeros(nb, np.int32)
    m = None if mass is None else np.ascontiguousarray(mass, dtype=np.float32)
    if m is not None and m.shape != idx.shape:
        raise ValueError("mass must have the shape of topk_idx")
    bad = lib().moe_oracle_coreset(_ptr(off), nb, R, E, k, _ptr(idx), _ptr(w), _ptr(m),
                                   ctypes.c_float(tau), _ptr(keep), _ptr(cs), _ptr(wr), _ptr(ne),
                                   int(max_experts))
    if bad < 0:
        raise ValueError("oracle coreset: invalid arguments")
    return keep, cs, wr, ne, int(bad)


def keep_mask(keep: np.ndarray, E: int) -> np.ndarray:
    """Bool [nb, E] view of the packed keep bits."""
    nb = keep.shape[0]
    out = np.zeros((nb, E), bool)
    for e in range(E):
        out[:, e] = (keep[:, e // 32] >> np.uint32(e % 32)) & 1
    return out


def dequant(q, d, bits):
    """Quantised weights back to bf16 bit patterns (reading 8 of moe_oracle.c: blocks
    of 32 along the input dimension, one bf16 scale each, weight = bf16(q * d)).

    q: int8 [..., rows, K] (bits 8) or uint8 [..., rows, K / 2] (bits 4, two per
    byte, even element in the low nibble); d: bf16 bits (uint16) [..., K / 32, rows].
    Returns uint16 [..., rows, K]."""
    q = np.ascontiguousarray(q)
    d = np.ascontiguousarray(d, dtype=np.uint16)
    lead = q.shape[:-2]
    rows = q.shape[-2]
    K = q.shape[-1] * (2 if bits == 4 else 1)
    out = np.zeros(lead + (rows, K), np.uint16)
    qf = q.reshape((-1,) + q.shape[-2:])
    df = d.reshape((-1,) + d.shape[-2:])
    of = out.reshape((-1, rows, K))
    for i in range(qf.shape[0]):
        qi, di = np.ascontiguousarray(qf[i]), np.ascontiguousarray(df[i])
        oi = np.zeros((rows, K), np.uint16)
        if lib().moe_oracle_dequant(_ptr(qi), _ptr(di), int(bits), rows, K, _ptr(oi)) != 0:
            raise ValueError("oracle dequant: invalid arguments")
        of[i] = oi
    return out


def expert_ffn(x_row, wg, wu, wd):
    """fp64 SwiGLU expert on one row: Wd (silu(Wg x) * (Wu x))."""
    x_row, wg, wu, wd = _u16(x_row), _u16(wg), _u16(wu), _u16(wd)
    I, H = wg.shape
    out = np.zeros(H, np.float64)
    lib().moe_oracle_expert_ffn(_ptr(x_row), _ptr(wg), _ptr(wu), _ptr(wd), H, I, _ptr(out))
    return out


def forward(x, block_offsets, topk_idx, w_renorm, keep, experts, shared, E, rows=None,
            nthreads=1):
    """y = shared(x) + sum over surviving pairs of w' * expert(x), in fp64.

    ``experts``: dict e -> (wg [I,H], wu [I,H], wd [H,I]) uint16 arrays; only the
    experts that surviving pairs use need to be present.  ``shared``: (sg, su, sd).
    ``rows``: optional sorted list of row indices to evaluate (others are 0).
    """
    x = _u16(x)
    R, H = x.shape
    off = np.ascontiguousarray(block_offsets, dtype=np.int32)
    nb = off.shape[0] - 1
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    wr = np.ascontiguousarray(w_renorm, dtype=np.float32)
    kp = np.ascontiguousarray(keep, dtype=np.uint32)
    k = idx.shape[1]
    sg, su, sd = (_u16(a) for a in shared)
    Is = sg.shape[0]
    I = next(iter(experts.values()))[0].shape[0] if experts else 1
    keepalive = []
    tabs = []
    for which in range(3):
        arr = (ctypes.c_void_p * E)()
        for e, mats in experts.items():
            m = _u16(mats[which])
            keepalive.append(m)
            arr[e] = m.ctypes.data
        tabs.append(arr)
    y = np.zeros((R, H), np.float64)
    if rows is None:
        rc = lib().moe_oracle_forward(_ptr(x), _ptr(off), nb, R, H, E, k, I, Is,
                                      ctypes.cast(tabs[0], ctypes.c_void_p),
                                      ctypes.cast(tabs[1], ctypes.c_void_p),
                                      ctypes.cast(tabs[2], ctypes.c_void_p),
                                      _ptr(sg), _ptr(su), _ptr(sd), _ptr(idx), _ptr(wr), _ptr(kp),
                                      _ptr(y), int(nthreads))
    else:
        # Evaluate a subset of rows: each as its own one-row block with its block's keep bits.
        bor = np.zeros(R, np.int64)
        for b in range(nb):
            bor[off[b]:off[b + 1]] = b
        rows = list(rows)
        xs = np.ascontiguousarray(x[rows])
        ids = np.ascontiguousarray(idx[rows])
        ws = np.ascontiguousarray(wr[rows])
        ks = np.ascontiguousarray(kp[bor[rows]])
        offs = np.arange(len(rows) + 1, dtype=np.int32)
        ys = np.zeros((len(rows), H), np.float64)
        rc = lib().moe_oracle_forward(_ptr(xs), _ptr(offs), len(rows), len(rows), H, E, k, I, Is,
                                      ctypes.cast(tabs[0], ctypes.c_void_p),
                                      ctypes.cast(tabs[1], ctypes.c_void_p),
                                      ctypes.cast(tabs[2], ctypes.c_void_p),
                                      _ptr(sg), _ptr(su), _ptr(sd), _ptr(ids), _ptr(ws), _ptr(ks),
                                      _ptr(ys), int(nthreads))
        y[rows] = ys
    if rc == -2:
        raise KeyError("oracle forward: a surviving pair uses an expert that was not supplied")
    if rc != 0:
        raise ValueError("oracle forward: invalid arguments")
    return y


def forward_live(x, block_offsets, topk_idx, w_renorm, keep, experts, shared, E, live, y_cached,
                 nthreads=1):
    """One live-row pass (InfiniLM PR #604, Summary and Motivation: live-row
    reuse with a refresh interval of five, neither defined there).  Reading:
    rows with live[r] != 0 get the expert FFN output of ``forward`` under the
    given keep mask; the others keep their cached output ``y_cached[r]``."""
    live = np.asarray(live)
    y = np.array(y_cached, dtype=np.float64, copy=True)
    rows = [int(r) for r in np.flatnonzero(live)]
    if rows:
        yl = forward(x, block_offsets, topk_idx, w_renorm, keep, experts, shared, E, rows=rows,
                     nthreads=nthreads)
        y[rows] = yl[rows]
    return y


def surviving_experts(topk_idx, keep, block_offsets, E):
    """Sorted list of experts used by at least one surviving (row, slot) pair."""
    mask = keep_mask(np.asarray(keep), E)
    off = np.asarray(block_offsets)
    used = set()
    for b in range(off.shape[0] - 1):
        ids = np.asarray(topk_idx)[off[b]:off[b + 1]].reshape(-1)
        for e in np.unique(ids):
            if 0 <= e < E and mask[b, e]:
                used.add(int(e))
    return sorted(used)
