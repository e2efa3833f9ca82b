"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol the public header declares, and rejects invalid arguments on the host
with a status and a message, before any CUDA work."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from sparse_moe_layer_row_gb300 import build as cbuild
from sparse_moe_layer_row_gb300 import moe_block as mb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return mb.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(moe_[a-z_0-9]+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("moe_block_route", "moe_block_coreset", "moe_block_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version(lib):
    assert mb.moe_version() >= 100


def dims(**kw):
    d = dict(H=2048, E=256, k=8, I=512, Is=512, max_rows=32, max_blocks=1)
    d.update(kw)
    return mb.moe_dims(**d)


def test_workspace_bytes_valid_and_monotone(lib):
    a = mb.moe_workspace_bytes(dims())
    b = mb.moe_workspace_bytes(dims(max_rows=8192, max_blocks=256))
    assert 0 < a < b
    assert a % 1024 == 0


@pytest.mark.parametrize("bad", [dict(H=0), dict(H=1000), dict(E=0), dict(E=1025), dict(k=0),
                                 dict(k=33), dict(E=4, k=5), dict(I=100), dict(Is=0),
                                 dict(max_rows=0), dict(max_blocks=0)], ids=str)
def test_workspace_bytes_rejects_bad_dims(lib, bad):
    assert mb.moe_workspace_bytes(dims(**bad)) == 0
    assert lib.moe_last_error().decode() != ""


def test_plan_create_rejects_null_and_misaligned_weights(lib):
    h = ctypes.c_void_p()
    rc = lib.moe_plan_create(ctypes.byref(dims()), *([None] * 7), ctypes.byref(h))
    assert rc == -1 and b"w_router" in lib.moe_last_error()
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(7)]
    ptrs[3] = ctypes.c_void_p(0x40008)
    rc = lib.moe_plan_create(ctypes.byref(dims()), *ptrs, ctypes.byref(h))
    assert rc == -1 and b"w_down" in lib.moe_last_error()
    rc = lib.moe_plan_create(ctypes.byref(dims(H=100)), *ptrs, ctypes.byref(h))
    assert rc == -2
    rc = lib.moe_plan_create(None, *ptrs, ctypes.byref(h))
    assert rc == -1


def test_calls_reject_null_plan(lib):
    ws = ctypes.c_void_p(0x100000)
    rc = lib.moe_block_route(None, ws, 4, ws, 1, None, ws, ws, ws, 1 << 20, None)
    assert rc == -1 and b"plan" in lib.moe_last_error()
    rc = lib.moe_block_coreset(None, 4, ws, 1, ws, ws, ctypes.c_float(0.9), ws, ws, ws, None, ws,
                               1 << 20, None)
    assert rc == -1
    rc = lib.moe_block_forward(None, ws, 4, ws, 1, ws, ws, ws, ws, None, ws, 1 << 20, None)
    assert rc == -1


def test_status_calls_reject_bad_workspace(lib):
    out = (ctypes.c_uint32 * 8)()
    assert lib.moe_read_device_status(None, None, out) == -1
    assert lib.moe_read_device_status(ctypes.c_void_p(0x100010), None, out) == -1
    assert lib.moe_clear_device_status(None, None) == -1


def test_binding_requires_cuda_tensors():
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mb._need(x, "x", torch.bfloat16, (4, 256))


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(mb, "_lib", None)
    monkeypatch.setattr(cbuild, "LIB", "/nonexistent/libmoeblock.so")
    with pytest.raises(ImportError):
        mb.load()


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_layer_row_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, re.M), f
                assert "moe_oracle" not in src, f


def test_live_pass_schedule():
    """Refresh every fifth pass: passes 0, 5, 10 evaluate every row (None)."""
    live = object()
    got = [mb.live_pass_mask(p, live) for p in range(11)]
    assert [g is None for g in got] == [p % 5 == 0 for p in range(11)]
    assert all(g is live for p, g in enumerate(got) if p % 5)
    assert mb.live_pass_mask(3, live, refresh=1) is None
    with pytest.raises(ValueError):
        mb.live_pass_mask(0, live, refresh=0)


def test_stack_dispatch_on_cpu():
    """MoeStack hands layer i its own input and bias (host logic, fake layers)."""
    calls = []

    class Fake:
        def __init__(self, i):
            self.i = i

        def __call__(self, x, off, tau, bias=None, stream=None, y=None):
            calls.append((self.i, x, bias, tau, y))
            return ("y", self.i) if y is None else y

    st = mb.MoeStack([Fake(0), Fake(1), Fake(2)])
    xs = [torch.zeros(1), torch.ones(1), torch.full((1,), 2.0)]
    outs = st(xs, torch.zeros(2, dtype=torch.int32), 0.9, biases=["b0", None, "b2"])
    assert outs == [("y", 0), ("y", 1), ("y", 2)]
    assert [c[0] for c in calls] == [0, 1, 2]
    assert all(c[1] is x for c, x in zip(calls, xs))
    assert [c[2] for c in calls] == ["b0", None, "b2"]
    calls.clear()
    one = torch.zeros(1)
    st(one, torch.zeros(2, dtype=torch.int32), 0.5)
    assert all(c[1] is one and c[2] is None for c in calls)
    with pytest.raises(ValueError):
        st(xs[:2], torch.zeros(2, dtype=torch.int32), 0.9)
    # given outputs go to the layers in order and come back
    calls.clear()
    ys = ["o0", "o1", "o2"]
    assert st(one, torch.zeros(2, dtype=torch.int32), 0.5, ys=ys) == ys
    assert [c[4] for c in calls] == ys
    with pytest.raises(ValueError):
        st(one, torch.zeros(2, dtype=torch.int32), 0.5, ys=ys[:1])
    with pytest.raises(ValueError):
        mb.MoeStack([])


def test_gate_up_interleave_layout():
    """The quantised gate/up tensor: rows 128 j .. 128 j + 63 are gate rows
    64 j .. 64 j + 63, the next 64 the up rows of the same indices, along the
    rows axis of codes (-2) and of block-major scales (-1); split inverts it."""
    from sparse_moe_layer_row_gb300 import workloads as W
    g = torch.arange(3 * 192 * 5).reshape(3, 192, 5)
    u = -1 - g
    t = W.interleave_gate_up(g, u, -2)
    assert t.shape == (3, 384, 5)
    for j in range(3):
        assert torch.equal(t[:, 128 * j:128 * j + 64], g[:, 64 * j:64 * j + 64])
        assert torch.equal(t[:, 128 * j + 64:128 * j + 128], u[:, 64 * j:64 * j + 64])
    g2, u2 = W.split_gate_up(t, -2)
    assert torch.equal(g2, g) and torch.equal(u2, u)
    s = W.interleave_gate_up(g.transpose(1, 2), u.transpose(1, 2), -1)
    assert torch.equal(s, t.transpose(1, 2))
    with pytest.raises(ValueError):
        W.interleave_gate_up(g[:, :96], u[:, :96], -2)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantised_experts_device_shapes(bits):
    """quantize_experts gives the shapes the quantised plan's tensor maps read,
    and gate_and_up(e) returns the per-matrix codes and scales it interleaved."""
    from sparse_moe_layer_row_gb300 import workloads as W
    w = W.TINY
    T = W.make_tensors(w)
    Q = W.quantize_experts(T, bits)
    kb = 1 if bits == 8 else 2
    assert Q.gate_up.shape == (w.E, 2 * w.I, w.H // kb)
    assert Q.gate_up_scale.shape == (w.E, w.H // 32, 2 * w.I)
    assert Q.shared_gate_up.shape == (2 * w.Is, w.H // kb)
    assert Q.shared_gate_up_scale.shape == (w.H // 32, 2 * w.Is)
    assert Q.down.shape == (w.E, w.H, w.I // kb) and Q.down_scale.shape == (w.E, w.I // 32, w.H)
    gq, gd, uq, ud = Q.gate_and_up(1)
    q, d = W.quantize_rows(T.w_gate[1], bits)
    assert torch.equal(gq, W.pack_int4(q) if bits == 4 else q)
    assert torch.equal(gd, W.scales_k_major(d))
    q, d = W.quantize_rows(T.w_up[1], bits)
    assert torch.equal(uq, W.pack_int4(q) if bits == 4 else q)
    assert torch.equal(ud, W.scales_k_major(d))
    # the binding's struct has the header's fields in the header's order
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "moe_block.h")).read()
    body = re.search(r"typedef struct moe_quant_weights \{(.*?)\}", hdr, re.S).group(1)
    assert re.findall(r"(\w+)\s*[,;]", body) == [f for f, _ in mb.moe_quant_weights._fields_]
