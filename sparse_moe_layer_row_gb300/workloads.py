"""Seeded synthetic workloads for the block-coreset MoE FFN.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It draws inputs and holds the workload shapes; it contains none of the
method's arithmetic (no routing, no coreset, no FFN).

Generator (counter-based, so any slice of any tensor can be drawn on its own,
on the CPU or on a CUDA device):

* ``splitmix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) as the mixing function;
* stream key ``K = mix(mix(seed) + tensor_id)``; element ``i`` uses the two
  words ``a = mix(K + 2i)`` and ``b = mix(K + 2i + 1)`` (all mod 2**64);
* ``u1 = ((a >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (b >> 11) * 2**-53``;
* Box-Muller in fp64: ``n = sqrt(-2 ln u1) * cos(2 pi u2)``;
* ``value = sigma * n`` rounded to bf16 (round-to-nearest-even by torch).

The workload shapes follow the model card "Clover-35B-A3B-Preview -- CMF"
(intro: 256 experts top-8 plus a shared expert, 32-token blocks; Usage: block
sizes 8/16/32 and a coreset carrying 90% of the block's routing).  Hidden and
intermediate sizes and value distributions are the synthetic stand-ins this
library is measured on; there are no trained weights.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB


def _signed(c: int) -> int:
    """uint64 constant -> the int64 with the same bits."""
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


def mix64_int(z: int) -> int:
    """splitmix64 finaliser on a Python int (exact uint64 arithmetic)."""
    z = (z + _GOLDEN) & _M64
    z = ((z ^ (z >> 30)) * _C1) & _M64
    z = ((z ^ (z >> 27)) * _C2) & _M64
    return z ^ (z >> 31)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_t(z: torch.Tensor) -> torch.Tensor:
    """splitmix64 on int64 tensors (two's-complement wrap = uint64 arithmetic)."""
    z = z + _signed(_GOLDEN)
    z = (z ^ _lsr(z, 30)) * _signed(_C1)
    z = (z ^ _lsr(z, 27)) * _signed(_C2)
    return z ^ _lsr(z, 31)


def stream_key(seed: int, tensor_id: int) -> int:
    return mix64_int((mix64_int(seed & _M64) + tensor_id) & _M64)


def uniform_words(seed: int, tensor_id: int, start: int, count: int,
                  device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """The raw word pair (a, b) of elements start..start+count-1 as int64 bits."""
    key = stream_key(seed, tensor_id)
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    base = idx * 2 + _signed(key)
    return _mix64_t(base), _mix64_t(base + 1)


def normal_f64(seed: int, tensor_id: int, start: int, count: int,
               device="cpu") -> torch.Tensor:
    a, b = uniform_words(seed, tensor_id, start, count, device)
    u1 = (_lsr(a, 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _lsr(b, 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal_bf16(seed: int, tensor_id: int, shape, sigma: float, device="cpu",
                start: int = 0, chunk: int = 1 << 26) -> torch.Tensor:
    """A bf16 tensor of ``shape`` whose flat element j is element start+j of the stream."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        v = normal_f64(seed, tensor_id, start + c0, c1 - c0, device) * sigma
        out[c0:c1] = v.to(torch.bfloat16)
    return out.view(*shape)


# Tensor ids inside one seed's family of streams.
TID_X, TID_WR, TID_WG, TID_WU, TID_WD, TID_SG, TID_SU, TID_SD, TID_PERM, TID_LIVE = range(1, 11)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, block layout, distributions and seeds."""
    name: str
    H: int
    E: int
    k: int
    I: int
    Is: int
    block_rows: tuple            # rows of each block, in order
    tau: float                   # coreset mass; >= 1 disables the coreset
    sigma_x: float = 1.0
    sigma_w: float = 0.02        # expert and shared-expert weights
    sigma_r: float = 0.02        # router weights
    zipf_s: float = 0.0          # > 0: per-block log-Zipf(s) logit bias
    x_seed: int = 0
    w_seed: int = 0
    description: str = ""

    @property
    def R(self) -> int:
        return int(sum(self.block_rows))

    @property
    def nb(self) -> int:
        return len(self.block_rows)

    def block_offsets(self) -> list:
        off = [0]
        for b in self.block_rows:
            off.append(off[-1] + int(b))
        return off

    def with_tau(self, tau: float, name: str | None = None) -> "Workload":
        return dataclasses.replace(self, tau=tau, name=name or f"{self.name}-tau{tau:g}")


# Weights of the full-shape configurations come from one fixed seed (one synthetic
# layer evaluated at several batch shapes); x and bias use the configuration's seed.
FULL_W_SEED = 1000

TINY = Workload(
    name="tiny-b32-h256-e16k4", H=256, E=16, k=4, I=128, Is=128, block_rows=(32,),
    tau=0.9, sigma_r=0.05, x_seed=0, w_seed=0,
    description="1 block of 32 rows, hidden 256, 16 experts top-4, intermediate 128")

BLOCK32 = Workload(
    name="block32-h2048-e256k8", H=2048, E=256, k=8, I=512, Is=512, block_rows=(32,),
    tau=0.9, x_seed=1, w_seed=FULL_W_SEED,
    description="one 32-row block, hidden 2048, 256 experts top-8, intermediate 512")

BLOCKS16_ZIPF = Workload(
    name="blocks16x32-zipf1.1", H=2048, E=256, k=8, I=512, Is=512, block_rows=(32,) * 16,
    tau=0.9, zipf_s=1.1, x_seed=2, w_seed=FULL_W_SEED,
    description="16 blocks of 32 rows with a per-block log-Zipf(1.1) expert preference")


def blocks2048(block: int, tau: float) -> Workload:
    return Workload(
        name=f"rows2048-b{block}-tau{tau:g}", H=2048, E=256, k=8, I=512, Is=512,
        block_rows=(block,) * (2048 // block), tau=tau, x_seed=3, w_seed=FULL_W_SEED,
        description=f"2048 rows in blocks of {block}, coreset mass {tau:g}")


ROWS2048 = tuple(blocks2048(b, t) for b in (32, 16, 8) for t in (0.9, 1.0))

PREFILL8192 = Workload(
    name="prefill8192-b32", H=2048, E=256, k=8, I=512, Is=512, block_rows=(32,) * 256,
    tau=0.9, x_seed=4, w_seed=FULL_W_SEED,
    description="256 blocks of 32 rows (8192 rows), uniform router")

ALL = (TINY, BLOCK32, BLOCKS16_ZIPF) + ROWS2048 + (PREFILL8192,)
BY_NAME = {w.name: w for w in ALL}


@dataclass
class Tensors:
    """Device-resident inputs of one workload."""
    x: torch.Tensor            # bf16 [R, H]
    w_router: torch.Tensor     # bf16 [E, H]
    w_gate: torch.Tensor       # bf16 [E, I, H]
    w_up: torch.Tensor         # bf16 [E, I, H]
    w_down: torch.Tensor       # bf16 [E, H, I]
    ws_gate: torch.Tensor      # bf16 [Is, H]
    ws_up: torch.Tensor        # bf16 [Is, H]
    ws_down: torch.Tensor      # bf16 [H, Is]
    bias: torch.Tensor | None  # fp32 [nb, E] or None
    block_offsets: torch.Tensor  # int32 [nb + 1]
    extra: dict = field(default_factory=dict)


def make_x(w: Workload, device="cpu", rows: int | None = None, seed: int | None = None):
    R = w.R if rows is None else rows
    s = w.x_seed if seed is None else seed
    return normal_bf16(s, TID_X, (R, w.H), w.sigma_x, device)


def make_router(w: Workload, device="cpu"):
    return normal_bf16(w.w_seed, TID_WR, (w.E, w.H), w.sigma_r, device)


def make_expert_slice(w: Workload, which: str, e0: int, e1: int, device="cpu"):
    """Experts e0..e1-1 of one routed weight tensor ('gate', 'up' or 'down')."""
    tid = {"gate": TID_WG, "up": TID_WU, "down": TID_WD}[which]
    per = w.I * w.H
    shape = (e1 - e0, w.I, w.H) if which != "down" else (e1 - e0, w.H, w.I)
    return normal_bf16(w.w_seed, tid, shape, w.sigma_w, device, start=e0 * per)


def make_shared(w: Workload, device="cpu"):
    g = normal_bf16(w.w_seed, TID_SG, (w.Is, w.H), w.sigma_w, device)
    u = normal_bf16(w.w_seed, TID_SU, (w.Is, w.H), w.sigma_w, device)
    d = normal_bf16(w.w_seed, TID_SD, (w.H, w.Is), w.sigma_w, device)
    return g, u, d


def zipf_bias(w: Workload, nb: int | None = None, seed: int | None = None) -> torch.Tensor | None:
    """Per-block logit bias: ln of the Zipf(s) pmf over a seeded random order of experts.

    Block b ranks the experts by the words of stream (seed, TID_PERM) at
    b*E .. b*E+E-1 (ascending, ties by id); the expert of rank j (1-based) gets
    ln(j**-s / sum_i i**-s).
    """
    if w.zipf_s <= 0:
        return None
    nb = w.nb if nb is None else nb
    s = w.x_seed if seed is None else seed
    E = w.E
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    logp = -w.zipf_s * torch.log(ranks)
    logp = logp - torch.log(torch.exp(logp).sum())
    bias = torch.empty(nb, E, dtype=torch.float32)
    for b in range(nb):
        a, _ = uniform_words(s, TID_PERM, b * E, E)
        key = _lsr(a, 1)  # non-negative 63-bit keys keep int64 order = uint64 order
        order = torch.argsort(key, stable=True)
        bias[b, order] = logp.to(torch.float32)
    return bias


def live_rows(R: int, frac: float, seed: int, device="cpu") -> torch.Tensor:
    """uint8 [R] row mask for live-row passes: row r is live (1) iff the top 53
    bits of word a of element r of stream (seed, TID_LIVE), as a fraction in
    [0, 1), fall below ``frac``."""
    a, _ = uniform_words(seed, TID_LIVE, 0, R)
    u = _lsr(a, 11).to(torch.float64) * (2.0 ** -53)
    return (u < frac).to(torch.uint8).to(device)


def make_tensors(w: Workload, device="cpu", x_seed: int | None = None) -> Tensors:
    x = make_x(w, device, seed=x_seed)
    wr = make_router(w, device)
    wg = make_expert_slice(w, "gate", 0, w.E, device)
    wu = make_expert_slice(w, "up", 0, w.E, device)
    wd = make_expert_slice(w, "down", 0, w.E, device)
    sg, su, sd = make_shared(w, device)
    bias = zipf_bias(w, seed=x_seed)
    if bias is not None:
        bias = bias.to(device)
    off = torch.tensor(w.block_offsets(), dtype=torch.int32, device=device)
    return Tensors(x, wr, wg, wu, wd, sg, su, sd, bias, off)


# --------------------------------------------------------------------------- quantised experts
#
# The 8-bit and 4-bit expert files of the model card ("Clover-35B-A3B-Preview
# -- CMF", Files: q8_2f, q4tp) store the experts in 8 and 4 bits; the page
# does not give the codecs.  The format used here: along each weight row's
# input dimension, blocks of 32 weights share one bf16 scale d; a weight is
# stored as a signed integer q (int8, or a 4-bit two's-complement nibble, two
# per byte, the even element in the low nibble) and stands for q * d rounded
# to bf16.  Synthetic quantised layers come from the synthetic bf16 layer by
# rounding to nearest (no calibration data): d = bf16(max|w| / qmax) per block,
# q = clamp(round(w / d)).  These functions only prepare inputs; the
# dequantisation itself belongs to each side (the kernels and the oracle).

QBLOCK = 32                   # weights per scale, along the input dimension
QMAX = {8: 127, 4: 7}


def quantize_rows(w: torch.Tensor, bits: int):
    """Round-to-nearest block quantisation of bf16 weights [..., rows, K].
    Returns (q int8 [..., rows, K] in [-qmax, qmax], d bf16 [..., rows, K / 32])."""
    if bits not in QMAX:
        raise ValueError("bits must be 8 or 4")
    *lead, rows, K = w.shape
    if K % QBLOCK:
        raise ValueError("the input dimension must be a multiple of 32")
    wf = w.float().reshape(*lead, rows, K // QBLOCK, QBLOCK)
    amax = wf.abs().amax(dim=-1)
    d = (amax / QMAX[bits]).to(torch.bfloat16)
    d = torch.where(d.float() > 0, d, torch.ones_like(d))   # all-zero block: any scale
    q = torch.round(wf / d.float().unsqueeze(-1)).clamp(-QMAX[bits], QMAX[bits]).to(torch.int8)
    return q.reshape(*lead, rows, K), d


def pack_int4(q: torch.Tensor) -> torch.Tensor:
    """int8 values in [-8, 7], last dim even -> uint8 with two per byte (element 2i
    in the low nibble, 2i + 1 in the high nibble, two's complement)."""
    u = (q.to(torch.int16) & 0xF).to(torch.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


def unpack_int4(p: torch.Tensor) -> torch.Tensor:
    """Inverse of pack_int4: uint8 [..., K/2] -> int8 [..., K]."""
    lo = (p & 0xF).to(torch.int16)
    hi = (p >> 4).to(torch.int16)
    lo = torch.where(lo >= 8, lo - 16, lo)
    hi = torch.where(hi >= 8, hi - 16, hi)
    out = torch.stack([lo, hi], dim=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    return out.to(torch.int8)


def scales_k_major(d: torch.Tensor) -> torch.Tensor:
    """Scales [..., rows, K/32] -> [..., K/32, rows] (the device layout: for one
    block of 32 along K, the scales of consecutive rows are contiguous)."""
    return d.transpose(-1, -2).contiguous()


GU_GROUP = 64   # gate and up rows interleave in groups of this many


def interleave_gate_up(g: torch.Tensor, u: torch.Tensor, axis: int) -> torch.Tensor:
    """Gate and up tensors (same shape) as one, their rows along ``axis``
    interleaved in groups of GU_GROUP: group j holds gate rows 64 j .. 64 j + 63,
    then the up rows of the same indices."""
    axis = axis % g.dim()
    n = g.shape[axis]
    if n % GU_GROUP:
        raise ValueError("the gate/up rows must be a multiple of 64")
    shp = list(g.shape)
    grouped = shp[:axis] + [n // GU_GROUP, 1, GU_GROUP] + shp[axis + 1:]
    both = torch.cat((g.reshape(grouped), u.reshape(grouped)), dim=axis + 1)
    return both.reshape(shp[:axis] + [2 * n] + shp[axis + 1:]).contiguous()


def split_gate_up(t: torch.Tensor, axis: int):
    """Inverse of interleave_gate_up: (gate, up)."""
    axis = axis % t.dim()
    n2 = t.shape[axis]
    shp = list(t.shape)
    grouped = t.reshape(shp[:axis] + [n2 // (2 * GU_GROUP), 2, GU_GROUP] + shp[axis + 1:])
    out = shp[:axis] + [n2 // 2] + shp[axis + 1:]
    return (grouped.select(axis + 1, 0).reshape(out).contiguous(),
            grouped.select(axis + 1, 1).reshape(out).contiguous())


@dataclass
class QuantExperts:
    """Quantised expert weights in the device layout.  Codes: int8 [E, rows, K] (8
    bits) or uint8 [E, rows, K / 2] (4 bits, packed); scales: bf16 [E, K / 32,
    rows].  The gate and up matrices are one tensor each for codes and scales, rows
    interleaved in groups of 64 (interleave_gate_up): gate_up [E, 2 I, K],
    gate_up_scale [E, K / 32, 2 I]; the shared expert's likewise."""
    bits: int
    gate_up: torch.Tensor
    down: torch.Tensor
    gate_up_scale: torch.Tensor
    down_scale: torch.Tensor
    shared_gate_up: torch.Tensor
    shared_down: torch.Tensor
    shared_gate_up_scale: torch.Tensor
    shared_down_scale: torch.Tensor

    def gate_and_up(self, e: int | None = None):
        """(gate codes, gate scales, up codes, up scales) of expert e, or of the
        shared expert (e None), each in the one-matrix layout."""
        if e is None:
            gq, uq = split_gate_up(self.shared_gate_up, -2)
            gd, ud = split_gate_up(self.shared_gate_up_scale, -1)
        else:
            gq, uq = split_gate_up(self.gate_up[e], -2)
            gd, ud = split_gate_up(self.gate_up_scale[e], -1)
        return gq, gd, uq, ud


def quantize_experts(T: "Tensors", bits: int) -> QuantExperts:
    """The routed and shared experts of `T` quantised (router untouched)."""
    def one(w):
        q, d = quantize_rows(w, bits)
        return (pack_int4(q) if bits == 4 else q.contiguous()), scales_k_major(d)
    (gq, gd), (uq, ud), (dq, dd), (sgq, sgd), (suq, sud), (sdq, sdd) = [
        one(w) for w in (T.w_gate, T.w_up, T.w_down, T.ws_gate, T.ws_up, T.ws_down)]
    return QuantExperts(bits, interleave_gate_up(gq, uq, -2), dq, interleave_gate_up(gd, ud, -1), dd,
                        interleave_gate_up(sgq, suq, -2), sdq, interleave_gate_up(sgd, sud, -1), sdd)
