"""Hand-worked fixtures under tests/golden/ (each file states its derivation and
the passage it follows): the oracle on CPU, and the CUDA coreset through the C
ABI on a GPU, against the values worked out by hand."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(values) -> np.ndarray:
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


CORESET = _load("coreset_hand.json")["cases"]
LOGITS = _load("logit_order_hand.json")["cases"]
FFN = _load("expert_ffn_hand.json")["cases"]


def _case_arrays(c):
    idx = np.array(c["topk_idx"], np.int32)
    wt = np.array(c["topk_w"], np.float32)
    return idx, wt


@pytest.fixture(scope="module")
def oracle_mod():
    import oracle
    return oracle


@pytest.mark.parametrize("c", CORESET, ids=lambda c: c["name"])
def test_oracle_coreset_hand_cases(oracle_mod, c):
    idx, wt = _case_arrays(c)
    keep, cs, wr, ne, _ = oracle_mod.coreset(c["block_offsets"], idx, wt, c["E"], c["tau"],
                                             max_experts=c["max_experts"])
    assert cs.tolist() == c["core_size"]
    assert keep[:, 0].tolist() == c["keep_bits"]
    assert np.array_equal(wr, np.array(c["w_renorm"], np.float32))
    assert ne.tolist() == c["n_empty"]


@pytest.mark.parametrize("c", LOGITS, ids=lambda c: c["name"])
def test_oracle_logit_order_hand_cases(oracle_mod, c):
    x = np.zeros(c["H"], np.float32)
    w = np.zeros(c["H"], np.float32)
    for h, xv, wv in c["products"]:
        x[h], w[h] = xv, wv
    assert oracle_mod.logit(_bf16_bits(x), _bf16_bits(w)) == c["logit"]


@pytest.mark.parametrize("c", FFN, ids=lambda c: c["name"])
def test_oracle_expert_ffn_hand_cases(oracle_mod, c):
    out = oracle_mod.expert_ffn(_bf16_bits(c["x"]), _bf16_bits(c["w_gate"]), _bf16_bits(c["w_up"]),
                                _bf16_bits(c["w_down"]))
    assert np.allclose(out, c["out"], rtol=1e-15, atol=1e-300)


def test_ffn_fixture_matches_its_derivation():
    """The fixture's numbers against the closed form in its derivation."""
    h = -1.0 / (1.0 + math.exp(-1.0))
    assert FFN[0]["out"] == [2 * h, -4 * h]


@pytest.mark.gpu
@pytest.mark.parametrize("c", CORESET, ids=lambda c: c["name"])
def test_cuda_coreset_hand_cases(c):
    """The CUDA coreset (k_coreset through moe_block_coreset / _budget) on the same
    hand-worked blocks: membership, sizes, weights and empty counts bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_layer_row_gb300 import moe_block
    dev = torch.device("cuda", 0)
    idx, wt = _case_arrays(c)
    R, k = idx.shape
    nb = len(c["block_offsets"]) - 1
    E, H, I = c["E"], 256, 64
    d = moe_block.moe_dims(H, E, k, I, I, R, nb)
    g = torch.Generator(device="cpu").manual_seed(1)

    def w(*shape):
        return (torch.randn(*shape, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    plan = moe_block.Plan(d, w(E, H), w(E, I, H), w(E, I, H), w(E, H, I), w(I, H), w(I, H), w(H, I))
    ws = plan.new_workspace()
    off = torch.tensor(c["block_offsets"], dtype=torch.int32, device=dev)
    keep = torch.empty(nb, (E + 31) // 32, dtype=torch.int32, device=dev)
    core = torch.empty(nb, dtype=torch.int32, device=dev)
    wr = torch.empty(R, k, dtype=torch.float32, device=dev)
    ne = torch.empty(nb, dtype=torch.int32, device=dev)
    moe_block.moe_block_coreset(plan, off, torch.from_numpy(idx).to(dev), torch.from_numpy(wt).to(dev),
                                c["tau"], keep, core, wr, ne, ws, max_experts=c["max_experts"])
    torch.cuda.synchronize()
    assert core.cpu().tolist() == c["core_size"]
    assert keep[:, 0].cpu().tolist() == c["keep_bits"]
    assert np.array_equal(wr.cpu().numpy(), np.array(c["w_renorm"], np.float32))
    assert ne.cpu().tolist() == c["n_empty"]


SOFTMAX = _load("softmax_sums_hand.json")


@pytest.mark.gpu
@pytest.mark.parametrize("c", SOFTMAX["cases"], ids=lambda c: c["name"])
def test_cuda_softmax_sums_hand_cases(c):
    """The CUDA router (moe_block_route_probs) on the hand-worked rows of
    softmax_sums_hand.json: the weight sum in rank order and the full-softmax
    denominator in lane order, bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from sparse_moe_layer_row_gb300 import moe_block
    dev = torch.device("cuda", 0)
    E, k, H, I = c["E"], c["k"], c["H"], 64
    wr = torch.zeros(E, H, dtype=torch.float32)
    wr[:, 0] = c["other_logit"]
    for e, z in c["logits"].items():
        wr[int(e), 0] = z
    x = torch.zeros(1, H, dtype=torch.float32)
    x[0, 0] = 1.0
    z = torch.zeros(E, I, H, dtype=torch.bfloat16, device=dev)
    zs = torch.zeros(I, H, dtype=torch.bfloat16, device=dev)
    plan = moe_block.Plan(moe_block.moe_dims(H, E, k, I, I, 1, 1), wr.to(torch.bfloat16).to(dev),
                          z, z, torch.zeros(E, H, I, dtype=torch.bfloat16, device=dev), zs, zs,
                          torch.zeros(H, I, dtype=torch.bfloat16, device=dev))
    ws = plan.new_workspace()
    idx = torch.empty(1, k, dtype=torch.int32, device=dev)
    w = torch.empty(1, k, dtype=torch.float32, device=dev)
    p = torch.empty(1, k, dtype=torch.float32, device=dev)
    off = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    moe_block.moe_block_route(plan, x.to(torch.bfloat16).to(dev), off, None, idx, w, ws, topk_p=p)
    torch.cuda.synchronize()
    delta = np.float32(oracle.exp_c(SOFTMAX["delta_arg"]))
    table = {"1": np.float32(1.0), "delta": delta, "1 - 2^-23": np.float32(1.0 - 2.0 ** -23),
             "delta / (1 + 2^-23)": np.float32(delta / np.float32(1.0 + 2.0 ** -23))}
    assert idx[0].cpu().tolist() == c["topk_idx"]
    want_w = np.array([table[e] for e in c["topk_w"]], np.float32)
    assert np.array_equal(w[0].cpu().numpy().view(np.uint32), want_w.view(np.uint32))
    if "topk_p" in c:
        want_p = np.array([table[e] for e in c["topk_p"]], np.float32)
        assert np.array_equal(p[0].cpu().numpy().view(np.uint32), want_p.view(np.uint32))
