"""Live-row reuse (InfiniLM PR #604, Summary and Motivation): a pass evaluates the
rows flagged live and leaves the cached output of the others.  The CUDA path
through the C ABI against the oracle on the same seeded inputs and mask: dead
rows untouched bit for bit, live rows equal to the full forward of the same
path bit for bit and to the oracle within the tolerance of parity_util."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.parity_util import Case, assert_close
from sparse_moe_layer_row_gb300 import moe_block, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    moe_block.load()


def _live_pass(case: Case, live: torch.Tensor):
    """Full forward (case.run), then a live-row pass into buffers holding a sentinel."""
    full = case.run()
    L = case.layer
    R, H, nb = case.R, case.w.H, case.nb
    idx, wr, keep = L._topk_idx[:R], L._w_renorm[:R], L._keep[:nb]
    g = torch.Generator(device="cpu").manual_seed(3)
    y32 = torch.randn(R, H, generator=g).to(case.dev)
    y = torch.randn(R, H, generator=g).to(torch.bfloat16).to(case.dev)
    y32_0, y_0 = y32.clone(), y.clone()
    L.forward(case.x, case.off, idx, wr, keep, y=y, y_f32=y32, live=live.to(case.dev))
    torch.cuda.synchronize()
    st = L.status()
    assert st["wait_timeout"] == 0
    return full, y, y32, y_0, y32_0


def _check(case: Case, live: torch.Tensor):
    full, y, y32, y_0, y32_0 = _live_pass(case, live)
    lv = live.bool().cpu().numpy()
    dead = ~lv
    # dead rows: not written
    assert torch.equal(y.cpu()[dead], y_0.cpu()[dead])
    assert torch.equal(y32.cpu()[dead], y32_0.cpu()[dead])
    # live rows: the full forward's values, bit for bit
    got32 = y32.cpu().numpy().astype(np.float64)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got32[lv], full["y32"][lv])
    assert np.array_equal(got[lv], full["y"][lv])
    # and the oracle's live-row pass on the live rows
    rows = np.flatnonzero(lv)
    if len(rows):
        case.oracle_route()
        case.oracle_coreset()
        yo = case.oracle_forward(rows=list(rows))
        assert_close(got32, yo, rows=rows, what="y_f32 (live rows)")
        assert_close(got, yo, rows=rows, what="y (live rows)")


@pytest.mark.parametrize("frac", [0.25, 0.7])
def test_live_rows_block32(frac):
    case = Case(W.BLOCK32)
    live = W.live_rows(case.R, frac, seed=21)
    assert 0 < int(live.sum()) < case.R
    _check(case, live)


def test_live_rows_zipf512():
    """16 blocks of 32 rows, per-block Zipf bias; a third of the rows live."""
    case = Case(W.BLOCKS16_ZIPF)
    _check(case, W.live_rows(case.R, 0.33, seed=22))


def test_live_rows_many_blocks_large_path():
    """2048 rows in blocks of 16 (large scatter, large GEMM shapes), 40% live."""
    case = Case(W.BY_NAME["rows2048-b16-tau0.9"])
    _check(case, W.live_rows(case.R, 0.4, seed=23))


def test_live_rows_prefill8192():
    """8192 rows (the prefill shape), 10% live: dead rows untouched, live rows equal
    the full forward bit for bit and match the oracle."""
    case = Case(W.PREFILL8192)
    _check(case, W.live_rows(case.R, 0.1, seed=24))


@pytest.mark.parametrize("wname", ["block32-h2048-e256k8", "rows2048-b32-tau0.9"])
def test_live_all_and_none(wname):
    case = Case(W.BY_NAME[wname])
    ones = torch.ones(case.R, dtype=torch.uint8)
    full, y, y32, _, _ = _live_pass(case, ones)
    assert np.array_equal(y32.cpu().numpy().astype(np.float64), full["y32"])
    zeros = torch.zeros(case.R, dtype=torch.uint8)
    _, y, y32, y_0, y32_0 = _live_pass(case, zeros)
    assert torch.equal(y, y_0) and torch.equal(y32, y32_0)


def test_live_single_row_ragged_blocks():
    """Ragged blocks (5, 32, 1, 26 rows): one live row in the last block."""
    w = W.BY_NAME["rows2048-b32-tau0.9"]
    T = W.make_tensors(w, device="cuda")
    off = [0, 5, 37, 38, 64]
    case = Case(w, T=T, block_offsets=off, bias=None, x=T.x[:64].contiguous())
    live = torch.zeros(64, dtype=torch.uint8)
    live[50] = 1
    _check(case, live)
