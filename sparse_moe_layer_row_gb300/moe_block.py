"""Python binding of libmoeblock (include/moe_block.h): argument marshalling only.

Every step of the layer runs in the CUDA kernels of the library; this module
checks tensor devices, dtypes and shapes, passes raw pointers and the current
CUDA stream through ctypes, and turns a non-OK status into an exception.
There is no CPU fallback: without the compiled library (or without a CUDA
device) every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MOE_OK = 0
STATUS_NAMES = ("nonfinite_logits", "bad_expert_id", "bad_offsets", "empty_rows", "wait_timeout",
                "nonfinite_output", "bad_unit")
STATUS_WORDS = 8


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"moe status {status}: {msg}")
        self.status = status


class moe_dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("Is", ctypes.c_int32), ("max_rows", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32)]


_QFIELDS = ("gate_up", "down", "gate_up_scale", "down_scale", "shared_gate_up", "shared_down",
            "shared_gate_up_scale", "shared_down_scale")


class moe_quant_weights(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32)] + [(n, ctypes.c_void_p) for n in _QFIELDS]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded libmoeblock.so.  Raises if it is not built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"libmoeblock.so is not built ({path}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        _build.build()
    L = ctypes.CDLL(path)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    L.moe_version.restype = i32
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_bytes.argtypes = [ctypes.POINTER(moe_dims)]
    L.moe_plan_create.restype = ctypes.c_int
    L.moe_plan_create.argtypes = [ctypes.POINTER(moe_dims), P, P, P, P, P, P, P,
                                  ctypes.POINTER(P)]
    L.moe_plan_create_quantized.restype = ctypes.c_int
    L.moe_plan_create_quantized.argtypes = [ctypes.POINTER(moe_dims), P,
                                            ctypes.POINTER(moe_quant_weights), ctypes.POINTER(P)]
    L.moe_plan_destroy.restype = None
    L.moe_plan_destroy.argtypes = [P]
    L.moe_block_route.restype = ctypes.c_int
    L.moe_block_route.argtypes = [P, P, i32, P, i32, P, P, P, P, sz, P]
    L.moe_block_coreset.restype = ctypes.c_int
    L.moe_block_coreset.argtypes = [P, i32, P, i32, P, P, ctypes.c_float, P, P, P, P, P, sz, P]
    L.moe_block_coreset_budget.restype = ctypes.c_int
    L.moe_block_coreset_budget.argtypes = [P, i32, P, i32, P, P, ctypes.c_float, i32, P, P, P, P, P,
                                           sz, P]
    L.moe_block_forward.restype = ctypes.c_int
    L.moe_block_forward.argtypes = [P, P, i32, P, i32, P, P, P, P, P, P, sz, P]
    L.moe_block_forward_live.restype = ctypes.c_int
    L.moe_block_forward_live.argtypes = [P, P, i32, P, i32, P, P, P, P, P, P, P, sz, P]
    L.moe_block_route_probs.restype = ctypes.c_int
    L.moe_block_route_probs.argtypes = [P, P, i32, P, i32, P, P, P, P, P, sz, P]
    L.moe_block_coreset_mass.restype = ctypes.c_int
    L.moe_block_coreset_mass.argtypes = [P, i32, P, i32, P, P, P, ctypes.c_float, i32, P, P, P,
                                         P, P, sz, P]
    L.moe_block_pass.restype = ctypes.c_int
    L.moe_block_pass.argtypes = [P, P, i32, P, i32, P, ctypes.c_float, i32, P, P, P, P, P, P, P,
                                 P, P, P, sz, P]
    L.moe_block_route_noalloc.restype = ctypes.c_int
    L.moe_block_route_noalloc.argtypes = [P, P, i32, P, i32, P, P, P, P]
    L.moe_plan_set_forward_events.restype = ctypes.c_int
    L.moe_plan_set_forward_events.argtypes = [P, P, i32]
    L.moe_plan_set_wait_limit.restype = ctypes.c_int
    L.moe_plan_set_wait_limit.argtypes = [P, ctypes.c_uint64]
    L.moe_read_device_status.restype = ctypes.c_int
    L.moe_read_device_status.argtypes = [P, P, P]
    L.moe_clear_device_status.restype = ctypes.c_int
    L.moe_clear_device_status.argtypes = [P, P]
    _lib = L
    return L


def _check(rc: int):
    if rc != MOE_OK:
        raise MoeError(rc, load().moe_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def moe_version() -> int:
    return int(load().moe_version())


def moe_workspace_bytes(dims: moe_dims) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(dims)))


class Plan:
    """moe_plan_create / moe_plan_destroy.  Keeps the weight tensors alive."""

    @classmethod
    def quantized(cls, dims: moe_dims, w_router, q):
        """moe_plan_create_quantized: ``q`` holds ``bits`` (8 or 4) and the codes and
        scales named as in moe_quant_weights (e.g. workloads.QuantExperts)."""
        d = dims
        bits = int(q.bits)
        if bits not in (8, 4):
            raise ValueError("bits must be 8 or 4")
        kb = 1 if bits == 8 else 2
        code = torch.int8 if bits == 8 else torch.uint8
        _need(w_router, "w_router", torch.bfloat16, (d.E, d.H))
        shapes = {"gate_up": (code, (d.E, 2 * d.I, d.H // kb)),
                  "down": (code, (d.E, d.H, d.I // kb)),
                  "gate_up_scale": (torch.bfloat16, (d.E, d.H // 32, 2 * d.I)),
                  "down_scale": (torch.bfloat16, (d.E, d.I // 32, d.H)),
                  "shared_gate_up": (code, (2 * d.Is, d.H // kb)),
                  "shared_down": (code, (d.H, d.Is // kb)),
                  "shared_gate_up_scale": (torch.bfloat16, (d.H // 32, 2 * d.Is)),
                  "shared_down_scale": (torch.bfloat16, (d.Is // 32, d.H))}
        tensors = [getattr(q, n) for n in _QFIELDS]
        for n, t in zip(_QFIELDS, tensors):
            _need(t, n, *shapes[n])
        self = cls.__new__(cls)
        self.dims = d
        self.weights = (w_router, *tensors)
        self.device = w_router.device
        self.bits = bits
        qw = moe_quant_weights(bits, *[t.data_ptr() for t in tensors])
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(load().moe_plan_create_quantized(ctypes.byref(d), _ptr(w_router),
                                                    ctypes.byref(qw), ctypes.byref(h)))
        self.handle = h
        return self

    def __init__(self, dims: moe_dims, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down):
        d = dims
        self.bits = 16
        _need(w_router, "w_router", torch.bfloat16, (d.E, d.H))
        _need(w_gate, "w_gate", torch.bfloat16, (d.E, d.I, d.H))
        _need(w_up, "w_up", torch.bfloat16, (d.E, d.I, d.H))
        _need(w_down, "w_down", torch.bfloat16, (d.E, d.H, d.I))
        _need(ws_gate, "ws_gate", torch.bfloat16, (d.Is, d.H))
        _need(ws_up, "ws_up", torch.bfloat16, (d.Is, d.H))
        _need(ws_down, "ws_down", torch.bfloat16, (d.H, d.Is))
        self.dims = d
        self.weights = (w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down)
        self.device = w_router.device
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(load().moe_plan_create(ctypes.byref(d), *[_ptr(w) for w in self.weights],
                                          ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            load().moe_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_forward_events(self, events):
        """Record 5 torch.cuda.Event(enable_timing=True) around the forward's kernels
        (before scatter, gate/up GEMM, down GEMM, final store; after the store).
        None turns the recording off."""
        if not events:
            _check(load().moe_plan_set_forward_events(self.handle, None, 0))
            self._events = None
            return
        if len(events) != 5:
            raise ValueError("need 5 events")
        for ev in events:
            if ev.cuda_event == 0:
                ev.record()  # torch creates the CUDA event lazily
        arr = (ctypes.c_void_p * 5)(*[ev.cuda_event for ev in events])
        _check(load().moe_plan_set_forward_events(self.handle, arr, 5))
        self._events = events

    def set_wait_limit(self, limit_ns: int):
        """moe_plan_set_wait_limit: the limit of the pipeline waits (0: built in).
        For tests of the failure path."""
        _check(load().moe_plan_set_wait_limit(self.handle, int(limit_ns)))

    def workspace_bytes(self) -> int:
        return moe_workspace_bytes(self.dims)

    def new_workspace(self) -> torch.Tensor:
        """A zeroed workspace (zero status counters)."""
        return torch.zeros(self.workspace_bytes(), dtype=torch.uint8, device=self.device)


def moe_block_route(plan: Plan, x, block_offsets, logit_bias, topk_idx, topk_w, workspace,
                    stream=None, topk_p=None):
    """moe_block_route, or moe_block_route_probs when ``topk_p`` (fp32 [R, k]) is given."""
    d = plan.dims
    R = x.shape[0]
    nb = block_offsets.shape[0] - 1
    _need(x, "x", torch.bfloat16, (R, d.H))
    _need(block_offsets, "block_offsets", torch.int32)
    if logit_bias is not None:
        _need(logit_bias, "logit_bias", torch.float32, (nb, d.E))
    _need(topk_idx, "topk_idx", torch.int32, (R, d.k))
    _need(topk_w, "topk_w", torch.float32, (R, d.k))
    _need(workspace, "workspace", torch.uint8)
    if topk_p is not None:
        _need(topk_p, "topk_p", torch.float32, (R, d.k))
        _check(load().moe_block_route_probs(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                            _ptr(logit_bias), _ptr(topk_idx), _ptr(topk_w),
                                            _ptr(topk_p), _ptr(workspace), workspace.numel(),
                                            _stream(stream)))
        return
    _check(load().moe_block_route(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                  _ptr(logit_bias), _ptr(topk_idx), _ptr(topk_w),
                                  _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_block_route_noalloc(plan: Plan, x, block_offsets, logit_bias, topk_idx, topk_w,
                            stream=None):
    """moe_block_route without a workspace, for callers that cannot allocate device
    memory: the scratch is a 1 MiB array inside the library (see the header for
    the size limit, and for why overlapping calls must not be issued)."""
    d = plan.dims
    R = x.shape[0]
    nb = block_offsets.shape[0] - 1
    _need(x, "x", torch.bfloat16, (R, d.H))
    _need(block_offsets, "block_offsets", torch.int32)
    if logit_bias is not None:
        _need(logit_bias, "logit_bias", torch.float32, (nb, d.E))
    _need(topk_idx, "topk_idx", torch.int32, (R, d.k))
    _need(topk_w, "topk_w", torch.float32, (R, d.k))
    _check(load().moe_block_route_noalloc(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                          _ptr(logit_bias), _ptr(topk_idx), _ptr(topk_w),
                                          _stream(stream)))


def moe_block_coreset(plan: Plan, block_offsets, topk_idx, topk_w, tau: float, keep, core_size,
                      w_renorm, n_empty, workspace, stream=None, max_experts: int = 0,
                      mass=None):
    """moe_block_coreset; moe_block_coreset_budget when max_experts != 0;
    moe_block_coreset_mass when ``mass`` (fp32 [R, k], e.g. topk_p) is given."""
    d = plan.dims
    R = topk_idx.shape[0]
    nb = block_offsets.shape[0] - 1
    _need(block_offsets, "block_offsets", torch.int32)
    _need(topk_idx, "topk_idx", torch.int32, (R, d.k))
    _need(topk_w, "topk_w", torch.float32, (R, d.k))
    _need(keep, "keep", torch.int32, (nb, (d.E + 31) // 32))
    _need(core_size, "core_size", torch.int32, (nb,))
    _need(w_renorm, "w_renorm", torch.float32, (R, d.k))
    if n_empty is not None:
        _need(n_empty, "n_empty", torch.int32, (nb,))
    _need(workspace, "workspace", torch.uint8)
    if mass is not None:
        _need(mass, "mass", torch.float32, (R, d.k))
        _check(load().moe_block_coreset_mass(plan.handle, R, _ptr(block_offsets), nb,
                                             _ptr(topk_idx), _ptr(topk_w), _ptr(mass),
                                             ctypes.c_float(tau), int(max_experts), _ptr(keep),
                                             _ptr(core_size), _ptr(w_renorm), _ptr(n_empty),
                                             _ptr(workspace), workspace.numel(), _stream(stream)))
        return
    if max_experts:
        _check(load().moe_block_coreset_budget(plan.handle, R, _ptr(block_offsets), nb,
                                               _ptr(topk_idx), _ptr(topk_w), ctypes.c_float(tau),
                                               int(max_experts), _ptr(keep), _ptr(core_size),
                                               _ptr(w_renorm), _ptr(n_empty), _ptr(workspace),
                                               workspace.numel(), _stream(stream)))
        return
    _check(load().moe_block_coreset(plan.handle, R, _ptr(block_offsets), nb, _ptr(topk_idx),
                                    _ptr(topk_w), ctypes.c_float(tau), _ptr(keep),
                                    _ptr(core_size), _ptr(w_renorm), _ptr(n_empty),
                                    _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_block_forward(plan: Plan, x, block_offsets, topk_idx, w_renorm, keep, y, y_f32, workspace,
                      stream=None, live=None):
    """Expert FFN of the pass.  ``live`` (uint8 [R], or None for every row)
    selects the rows evaluated; the others keep what ``y`` / ``y_f32`` hold."""
    d = plan.dims
    R = x.shape[0]
    nb = block_offsets.shape[0] - 1
    _need(x, "x", torch.bfloat16, (R, d.H))
    _need(block_offsets, "block_offsets", torch.int32)
    _need(topk_idx, "topk_idx", torch.int32, (R, d.k))
    _need(w_renorm, "w_renorm", torch.float32, (R, d.k))
    _need(keep, "keep", torch.int32, (nb, (d.E + 31) // 32))
    _need(y, "y", torch.bfloat16, (R, d.H))
    if y_f32 is not None:
        _need(y_f32, "y_f32", torch.float32, (R, d.H))
    _need(workspace, "workspace", torch.uint8)
    if live is not None:
        _need(live, "live", torch.uint8, (R,))
        _check(load().moe_block_forward_live(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                             _ptr(topk_idx), _ptr(w_renorm), _ptr(keep),
                                             _ptr(live), _ptr(y), _ptr(y_f32), _ptr(workspace),
                                             workspace.numel(), _stream(stream)))
        return
    _check(load().moe_block_forward(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                    _ptr(topk_idx), _ptr(w_renorm), _ptr(keep), _ptr(y),
                                    _ptr(y_f32), _ptr(workspace), workspace.numel(),
                                    _stream(stream)))


def moe_block_pass(plan: Plan, x, block_offsets, logit_bias, tau: float, max_experts: int,
                   topk_idx, topk_w, topk_p, keep, core_size, w_renorm, n_empty, y, y_f32,
                   workspace, stream=None):
    """One pass: route -> coreset -> forward in one call.
    ``topk_p`` None: the weight mass; a tensor: the probability mass."""
    d = plan.dims
    R = x.shape[0]
    nb = block_offsets.shape[0] - 1
    _need(x, "x", torch.bfloat16, (R, d.H))
    _need(block_offsets, "block_offsets", torch.int32)
    if logit_bias is not None:
        _need(logit_bias, "logit_bias", torch.float32, (nb, d.E))
    _need(topk_idx, "topk_idx", torch.int32, (R, d.k))
    _need(topk_w, "topk_w", torch.float32, (R, d.k))
    if topk_p is not None:
        _need(topk_p, "topk_p", torch.float32, (R, d.k))
    _need(keep, "keep", torch.int32, (nb, (d.E + 31) // 32))
    _need(core_size, "core_size", torch.int32, (nb,))
    _need(w_renorm, "w_renorm", torch.float32, (R, d.k))
    if n_empty is not None:
        _need(n_empty, "n_empty", torch.int32, (nb,))
    _need(y, "y", torch.bfloat16, (R, d.H))
    if y_f32 is not None:
        _need(y_f32, "y_f32", torch.float32, (R, d.H))
    _need(workspace, "workspace", torch.uint8)
    _check(load().moe_block_pass(plan.handle, _ptr(x), R, _ptr(block_offsets), nb,
                                 _ptr(logit_bias), ctypes.c_float(tau), int(max_experts),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(topk_p), _ptr(keep),
                                 _ptr(core_size), _ptr(w_renorm), _ptr(n_empty), _ptr(y),
                                 _ptr(y_f32), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))


def moe_read_device_status(workspace: torch.Tensor, stream=None) -> dict:
    _need(workspace, "workspace", torch.uint8)
    out = (ctypes.c_uint32 * STATUS_WORDS)()
    _check(load().moe_read_device_status(_ptr(workspace), _stream(stream), out))
    return {name: int(out[i]) for i, name in enumerate(STATUS_NAMES)}


def moe_clear_device_status(workspace: torch.Tensor, stream=None):
    _need(workspace, "workspace", torch.uint8)
    _check(load().moe_clear_device_status(_ptr(workspace), _stream(stream)))


def live_pass_mask(pass_index: int, live, refresh: int = 5):
    """Live-row reuse schedule (InfiniLM PR #604, Summary and Motivation: refresh
    interval five).  Pass 0 and every ``refresh``-th pass after it evaluate every
    row (returns None); the passes between evaluate the rows of ``live`` only."""
    if refresh < 1:
        raise ValueError("refresh interval must be >= 1")
    if pass_index < 0:
        raise ValueError("pass index must be >= 0")
    return None if pass_index % refresh == 0 else live


SMALL_ROWS = 32   # calls of at most this many rows take the weight-streaming kernels


class MoeBlockLayer:
    """The whole pass: route -> coreset -> forward, with its own workspace and buffers.

    Weights are the seven bf16 tensors of moe_plan_create; ``max_rows`` and
    ``max_blocks`` size the workspace.  ``__call__`` enqueues three C-ABI calls
    on the current stream and returns y (bf16 [R, H]).
    """

    def __init__(self, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, k: int,
                 max_rows: int, max_blocks: int, plan=None):
        E, H = w_router.shape
        I = w_gate.shape[1]
        Is = ws_gate.shape[0]
        self.dims = moe_dims(H, E, k, I, Is, max_rows, max_blocks)
        self.plan = plan if plan is not None else Plan(self.dims, w_router, w_gate, w_up, w_down,
                                                       ws_gate, ws_up, ws_down)
        self._init_buffers(w_router.device)

    @classmethod
    def quantized(cls, w_router, q, k: int, max_rows: int, max_blocks: int):
        """A layer whose experts are quantised (moe_plan_create_quantized; ``q`` as
        for Plan.quantized, e.g. workloads.QuantExperts)."""
        E, H = w_router.shape
        I = q.gate_up_scale.shape[-1] // 2
        Is = q.shared_gate_up_scale.shape[-1] // 2
        self = cls.__new__(cls)
        self.dims = moe_dims(H, E, k, I, Is, max_rows, max_blocks)
        self.plan = Plan.quantized(self.dims, w_router, q)
        self._init_buffers(w_router.device)
        return self

    def _init_buffers(self, dev):
        E, H, k = self.dims.E, self.dims.H, self.dims.k
        max_rows, max_blocks = self.dims.max_rows, self.dims.max_blocks
        self.workspace = self.plan.new_workspace()
        R, nb, words = max_rows, max_blocks, (E + 31) // 32
        self._topk_idx = torch.empty(R, k, dtype=torch.int32, device=dev)
        self._topk_w = torch.empty(R, k, dtype=torch.float32, device=dev)
        self._w_renorm = torch.empty(R, k, dtype=torch.float32, device=dev)
        self._keep = torch.empty(nb, words, dtype=torch.int32, device=dev)
        self._core = torch.empty(nb, dtype=torch.int32, device=dev)
        self._empty = torch.empty(nb, dtype=torch.int32, device=dev)
        self._y = torch.empty(R, H, dtype=torch.bfloat16, device=dev)

    def route(self, x, block_offsets, bias=None, stream=None, probs=False):
        """Returns (topk_idx, topk_w), and topk_p as a third value with ``probs``."""
        R = x.shape[0]
        idx, w = self._topk_idx[:R], self._topk_w[:R]
        if probs:
            if not hasattr(self, "_topk_p"):
                self._topk_p = torch.empty_like(self._topk_w)
            p = self._topk_p[:R]
            moe_block_route(self.plan, x, block_offsets, bias, idx, w, self.workspace, stream,
                            topk_p=p)
            return idx, w, p
        moe_block_route(self.plan, x, block_offsets, bias, idx, w, self.workspace, stream)
        return idx, w

    def coreset(self, block_offsets, topk_idx, topk_w, tau, stream=None, max_experts=0,
                mass=None):
        R = topk_idx.shape[0]
        nb = block_offsets.shape[0] - 1
        keep, core, empty = self._keep[:nb], self._core[:nb], self._empty[:nb]
        wr = self._w_renorm[:R]
        moe_block_coreset(self.plan, block_offsets, topk_idx, topk_w, tau, keep, core, wr, empty,
                          self.workspace, stream, max_experts=max_experts, mass=mass)
        return keep, core, wr, empty

    def forward(self, x, block_offsets, topk_idx, w_renorm, keep, y=None, y_f32=None,
                stream=None, live=None):
        R = x.shape[0]
        y = self._y[:R] if y is None else y
        moe_block_forward(self.plan, x, block_offsets, topk_idx, w_renorm, keep, y, y_f32,
                          self.workspace, stream, live=live)
        return y

    def __call__(self, x, block_offsets, tau: float, bias=None, y=None, y_f32=None, stream=None,
                 max_experts: int = 0, probs: bool = False):
        """One pass (moe_block_pass): route -> coreset -> forward; returns y.  The
        routing outputs stay in the layer's buffers (topk_idx, topk_w, keep,
        w_renorm ...) until the next call."""
        R = x.shape[0]
        nb = block_offsets.shape[0] - 1
        y = self._y[:R] if y is None else y
        p = None
        if probs:
            if not hasattr(self, "_topk_p"):
                self._topk_p = torch.empty_like(self._topk_w)
            p = self._topk_p[:R]
        moe_block_pass(self.plan, x, block_offsets, bias, tau, max_experts, self._topk_idx[:R],
                       self._topk_w[:R], p, self._keep[:nb], self._core[:nb], self._w_renorm[:R],
                       self._empty[:nb], y, y_f32, self.workspace, stream)
        return y

    def status(self, stream=None) -> dict:
        return moe_read_device_status(self.workspace, stream)


class MoeStack:
    """Several MoE layers of one pass, enqueued back to back on one stream with
    no host synchronisation, so that ``capture`` can record the whole pass as
    one CUDA graph and a replay submits it as one launch (model card
    "Clover-35B-A3B-Preview -- CMF", Hardware: every pass as one GPU submission).
    Layer i reads ``xs[i]``: what a model computes between its MoE layers
    (attention, norms, the residual stream) is the caller's, and its kernels can
    be captured into the same graph around these calls.
    """

    def __init__(self, layers):
        self.layers = list(layers)
        if not self.layers:
            raise ValueError("a stack needs at least one layer")

    def __call__(self, xs, block_offsets, tau: float, biases=None, stream=None, ys=None):
        """Runs every layer on its input (``xs``: one tensor per layer, or one
        tensor for all) and returns the layers' outputs: ``ys`` (one bf16 [R, H]
        tensor per layer) when given, else each layer's own output buffer, which
        the layer's next call overwrites."""
        if isinstance(xs, torch.Tensor):
            xs = [xs] * len(self.layers)
        if len(xs) != len(self.layers):
            raise ValueError("one input per layer")
        if ys is not None and len(ys) != len(self.layers):
            raise ValueError("one output per layer")
        return [layer(x, block_offsets, tau, bias=None if biases is None else biases[i],
                      stream=stream, y=None if ys is None else ys[i])
                for i, (layer, x) in enumerate(zip(self.layers, xs))]

    def capture(self, xs, block_offsets, tau: float, biases=None):
        """Record one pass over the static inputs ``xs`` as a CUDA graph.  Returns
        (graph, outputs); ``graph.replay()`` reruns the pass on whatever the inputs
        and ``block_offsets`` then hold and rewrites ``outputs`` in place.  The
        outputs are tensors of the graph's own, so eager calls of the same layers
        (or other graphs over them) do not overwrite them; the layers' workspaces
        are shared, so replays and eager calls of the same layers must not run
        concurrently."""
        dev = block_offsets.device
        outs = []
        xl = [xs] * len(self.layers) if isinstance(xs, torch.Tensor) else list(xs)
        for layer, x in zip(self.layers, xl):
            outs.append(torch.empty(x.shape[0], layer.dims.H, dtype=torch.bfloat16, device=dev))
        stream = torch.cuda.Stream(device=dev)
        stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(stream):
            self(xs, block_offsets, tau, biases, ys=outs)   # warm-up outside the capture
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self(xs, block_offsets, tau, biases, ys=outs)
        torch.cuda.current_stream(dev).wait_stream(stream)
        return graph, outs
