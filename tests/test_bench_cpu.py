"""Host logic of bench.py (no GPU): the algorithmic accounting, the roofline
summary of a measurement, and which workloads share the layer's weights."""
from __future__ import annotations

import math

import pytest
import torch

import bench
from sparse_moe_layer_row_gb300 import workloads as W

PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="test")


def test_accounting_full_shape_block():
    w = W.BLOCK32
    a = bench.accounting(w, 32, 122, 223)
    expert = 3 * 2048 * 512 * 2
    assert a["step_bytes"] == 122 * expert + expert + 256 * 2048 * 2 + 2 * 32 * 2048 * 2
    assert a["gu_bytes"] == 122 * 2 * 2048 * 512 * 2 + 2 * 2048 * 512 * 2 + 32 * 2048 * 2
    assert a["step_flops"] == 2.0 * 32 * 2048 * 256 + 223 * 6.0 * 2048 * 512 + 32 * 6.0 * 2048 * 512
    assert a["gu_flops"] == 4.0 * 2048 * (223 * 512 + 32 * 512)


def _meas(w, used, pairs, step_ms, gu_ms):
    return dict(total_ms=step_ms * 10, steps=10, used=set(range(used)), pairs=pairs,
                kern={"front": [0.01], "gate_up": [gu_ms], "down": [0.02], "combine": [0.005]},
                phase_ms={"route": [0.01], "coreset": [0.01], "forward": [0.1]}, clocks=None)


def test_summarize_hbm_bound_block():
    w = W.BLOCK32
    s = bench.summarize(w, _meas(w, 122, 223, 0.176, 0.085), PEAKS)
    acc = bench.accounting(w, 32, 122, 223)
    assert s["roofline"]["bound"] == "hbm" and s["roofline"]["unit"] == "GB/s"
    assert math.isclose(s["roofline"]["achieved"], acc["gu_bytes"] / 85e-6 / 1e9)
    assert math.isclose(s["roofline"]["frac"], s["roofline"]["achieved"] / 6800.0)
    assert math.isclose(s["value"], 32 * 10 / (1.76e-3))
    assert math.isclose(s["step_roofline_frac"], acc["step_bytes"] / 6800e9 / 176e-6)
    assert s["step_roofline_bound"] == "hbm"
    assert set(s["kernel_us"]) == {"front", "gate_up", "down", "combine"}


def test_summarize_binding_roof():
    """The gate/up roofline is the tighter roof: the larger of the kernel's HBM
    time and its tensor time at the measured peaks."""
    w = W.PREFILL8192
    # 56,651 pairs over 256 experts: 1.11 GB at 6.8 TB/s (164 us) outlasts
    # 272 GFLOP at 1.9 PFLOP/s (143 us), so HBM binds
    s = bench.summarize(w, _meas(w, 256, 56651, 0.65, 0.26), PEAKS)
    acc = bench.accounting(w, 8192, 256, 56651)
    assert acc["gu_bytes"] / 6800e9 > acc["gu_flops"] / 1900e12
    assert s["roofline"]["bound"] == "hbm" and s["roofline"]["unit"] == "GB/s"
    assert math.isclose(s["roofline"]["achieved"], acc["gu_bytes"] / 0.26e-3 / 1e9)
    assert math.isclose(s["roofline"]["tflops_alongside"], acc["gu_flops"] / 0.26e-3 / 1e12)
    # four times the pairs: the FLOPs bind
    s = bench.summarize(w, _meas(w, 256, 4 * 56651, 0.65, 0.5), PEAKS)
    acc = bench.accounting(w, 8192, 256, 4 * 56651)
    assert acc["gu_flops"] / 1900e12 > acc["gu_bytes"] / 6800e9
    assert s["roofline"]["bound"] == "tensor" and s["roofline"]["unit"] == "TFLOP/s"
    assert math.isclose(s["roofline"]["achieved"], acc["gu_flops"] / 0.5e-3 / 1e12)
    assert s["roofline"]["frac"] == pytest.approx(s["roofline"]["achieved"] / 1900.0)


def test_extra_workloads_share_the_layer():
    dev = torch.device("cpu")
    w = W.TINY
    T = W.make_tensors(w)
    same = bench.tensors_like(w, w, T, dev, x_seed=5)
    assert same.w_gate is T.w_gate and same.x.shape == T.x.shape
    assert not torch.equal(same.x, T.x)
    for name in bench.EXTRA_WORKLOADS:
        we = W.BY_NAME[name]
        assert (we.H, we.E, we.w_seed) == (W.BLOCK32.H, W.BLOCK32.E, W.BLOCK32.w_seed)
