"""Pins of the CPU oracle against facts that do not come from the oracle itself.

The pages print no worked example for the MoE layer, so the oracle is pinned by
hand-derived values, closed forms, exhaustive enumeration on tiny expert counts,
invariants the method must satisfy, and the special case tau >= 1 (coreset
disabled = plain top-k MoE, InfiniLM PR #604, Notes: full-route replay).
"""
from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from sparse_moe_layer_row_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_bits(vals) -> np.ndarray:
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    t = torch.tensor(vals, dtype=torch.float32)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "value not exactly representable in bf16"
    return u16(b)


def f32(x) -> float:
    return float(np.float32(x))


def ulp32(x: float) -> float:
    x = abs(np.float32(x))
    return float(np.spacing(x)) if x > 0 else float(np.spacing(np.float32(0)))


# --------------------------------------------------------------------------- generator

def test_generator_is_splitmix64_definition():
    """The int64 tensor implementation equals exact uint64 arithmetic on Python ints."""
    for seed, tid in [(0, 1), (1000, 5), (123456789, 9)]:
        key = W.stream_key(seed, tid)
        for start in (0, 17, (1 << 33) + 5):
            a, b = W.uniform_words(seed, tid, start, 64)
            for i in range(64):
                ea = W.mix64_int((key + 2 * (start + i)) & W._M64)
                eb = W.mix64_int((key + 2 * (start + i) + 1) & W._M64)
                assert int(a[i]) & W._M64 == ea
                assert int(b[i]) & W._M64 == eb


def test_generator_known_splitmix_value():
    # splitmix64 with state 0: first output is 0xE220A8397B1DCDAF (published test vector)
    assert W.mix64_int(0) == 0xE220A8397B1DCDAF


def test_generator_slices_and_moments():
    full = W.normal_bf16(7, 3, (4, 1000), 0.5)
    part = W.normal_bf16(7, 3, (2, 1000), 0.5, start=2000)
    assert torch.equal(full[2:], part)
    v = W.normal_f64(7, 3, 0, 200000)
    assert abs(float(v.mean())) < 0.01 and abs(float(v.std()) - 1.0) < 0.01


def test_zipf_bias_is_log_pmf_permutation():
    w = W.BLOCKS16_ZIPF
    b = W.zipf_bias(w)
    assert b.shape == (16, 256)
    for r in range(16):
        p = torch.exp(b[r].double())
        assert abs(float(p.sum()) - 1.0) < 1e-5
        sorted_vals = torch.sort(b[r], descending=True).values.double()
        ranks = torch.arange(1, 257, dtype=torch.float64)
        expect = -1.1 * torch.log(ranks)
        expect -= torch.log(torch.exp(expect).sum())
        assert torch.allclose(sorted_vals, expect, atol=1e-5)
    assert not torch.equal(b[0], b[1])


# --------------------------------------------------------------------------- exp_c

def test_exp_c_special_values(oracle_mod):
    assert oracle_mod.exp_c(0.0) == 1.0
    assert oracle_mod.exp_c(-0.0) == 1.0
    assert oracle_mod.exp_c(-87.5) == 0.0
    assert oracle_mod.exp_c(-1e30) == 0.0
    assert oracle_mod.exp_c(float("-inf")) == 0.0
    assert oracle_mod.exp_c(float("nan")) == 0.0


def test_exp_c_within_two_ulp_of_exp(oracle_mod):
    """exp_c is within 2 ulp of the correctly rounded exponential on [-87, 0]."""
    rng = np.random.default_rng(0)
    ts = np.concatenate([np.linspace(-87.0, 0.0, 20001), -rng.exponential(3.0, 20000),
                         -np.logspace(-8, 1.9, 2000)]).astype(np.float32)
    ts = ts[ts >= -87.0]
    worst = 0.0
    for t in ts:
        got = oracle_mod.exp_c(float(t))
        ref = math.exp(float(t))
        err = abs(got - ref) / ulp32(f32(ref))
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_exp_c_is_monotone_on_grid(oracle_mod):
    ts = np.linspace(-20.0, 0.0, 4001).astype(np.float32)
    vals = [oracle_mod.exp_c(float(t)) for t in ts]
    assert all(a <= b for a, b in zip(vals, vals[1:]))


# --------------------------------------------------------------------------- logits

def _logit_pair(H, products_at):
    """x, w rows with x[h]*w[h] = given exact products at chosen positions, 0 elsewhere."""
    x = np.zeros(H, np.float32)
    w = np.zeros(H, np.float32)
    for h, (a, b) in products_at.items():
        x[h], w[h] = a, b
    return bf16_bits(x), bf16_bits(w)


def test_logit_lane_order_hand_value(oracle_mod):
    """Lane 0 owns h = 0..7 and adds in ascending h: (2^24 + 1) - 2^24 = 0 in fp32
    (2^24 + 1 rounds to even, 2^24), while the exact dot product is 1."""
    x, w = _logit_pair(256, {0: (4096.0, 4096.0), 1: (1.0, 1.0), 2: (-4096.0, 4096.0)})
    assert oracle_mod.logit(x, w) == 0.0
    # lane 1 (h = 8..15): 2^24 - 2^24 first, then + 1: the 1 survives
    x, w = _logit_pair(256, {8: (4096.0, 4096.0), 9: (-4096.0, 4096.0), 10: (1.0, 1.0)})
    assert oracle_mod.logit(x, w) == 1.0


def test_logit_butterfly_hand_value(oracle_mod):
    """Partial sums s_0 = 2^24, s_16 = 1, s_8 = -2^24: the xor butterfly adds lanes
    0+16 first (2^24 + 1 -> 2^24), then (0,16)+(8,24) -> 0; a sequential lane sum
    would give 1."""
    x, w = _logit_pair(256, {0: (4096.0, 4096.0), 128: (1.0, 1.0), 64: (-4096.0, 4096.0)})
    assert oracle_mod.logit(x, w) == 0.0
    # lane 1 (h=8) with lane 0: step o=1 pairs them last, after 16/8/4/2
    x, w = _logit_pair(256, {0: (4096.0, 4096.0), 8: (-4096.0, 4096.0), 128: (1.0, 1.0)})
    # o=16: lane0 = 2^24 + 1 -> 2^24; lane1 = -2^24 + 0; ... o=1: 2^24 - 2^24 = 0
    assert oracle_mod.logit(x, w) == 0.0


def test_logit_stripe_order_hand_value(oracle_mod):
    """Lane 0's elements of stripe 0 come before those of stripe 1 (h = 256)."""
    x, w = _logit_pair(512, {0: (4096.0, 4096.0), 1: (1.0, 1.0), 256: (-4096.0, 4096.0)})
    assert oracle_mod.logit(x, w) == 0.0
    # stripe 0 cancels to 0 before stripe 1 adds 1 (stripe 1 first would lose the 1)
    x, w = _logit_pair(512, {0: (4096.0, 4096.0), 1: (-4096.0, 4096.0), 256: (1.0, 1.0)})
    assert oracle_mod.logit(x, w) == 1.0


def test_logit_within_summation_bound(oracle_mod):
    """|z - z_exact| <= gamma_n * sum|x w|, n = H/32 + 5 (recursive summation bound)."""
    w = W.BLOCK32
    x = u16(W.make_x(w, rows=4))
    wr = u16(W.make_router(w))
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    wf = torch.from_numpy(wr.view(np.int16)).view(torch.bfloat16).double().numpy()
    u = 2.0 ** -24
    n = w.H // 32 + 5
    gamma = n * u / (1 - n * u)
    for r in range(4):
        for e in range(0, 256, 7):
            z = oracle_mod.logit(x[r], wr[e])
            exact = float(np.dot(xf[r], wf[e]))
            bound = gamma * float(np.abs(xf[r] * wf[e]).sum())
            assert abs(z - exact) <= bound


def test_route_logits_match_single_logit_and_bias(oracle_mod):
    w = W.TINY
    T = W.make_tensors(w)
    x, wr = u16(T.x), u16(T.w_router)
    bias = np.linspace(-1, 1, w.E, dtype=np.float32)[None, :]
    idx, wt, z, nf = oracle_mod.route(x, wr, [0, w.R], w.k, bias=bias, want_logits=True)
    assert nf == 0
    for r in range(0, w.R, 5):
        for e in range(w.E):
            assert z[r, e] == np.float32(np.float32(oracle_mod.logit(x[r], wr[e])) + bias[0, e])


# --------------------------------------------------------------------------- top-k + weights

def test_topk_is_sorted_selection(oracle_mod):
    w = W.BLOCK32
    x = u16(W.make_x(w))
    wr = u16(W.make_router(w))
    idx, wt, z, nf = oracle_mod.route(x, wr, w.block_offsets(), w.k, want_logits=True)
    for r in range(w.R):
        sel = list(idx[r])
        assert len(set(sel)) == w.k
        keyed = sorted(range(w.E), key=lambda e: (-float(z[r, e]), e))
        assert sel == keyed[:w.k]


def test_topk_ties_go_to_lower_id(oracle_mod):
    """Experts with identical router rows have equal logits; the lower id ranks first."""
    w = W.TINY
    T = W.make_tensors(w)
    wr = T.w_router.clone()
    wr[9] = wr[2]
    wr[14] = wr[2]
    x = u16(T.x)
    idx, wt, z, nf = oracle_mod.route(x, u16(wr), [0, w.R], w.k, want_logits=True)
    hit = 0
    for r in range(w.R):
        assert z[r, 2] == z[r, 9] == z[r, 14]
        row = list(idx[r])
        pos = [row.index(e) for e in (2, 9, 14) if e in row]
        assert pos == sorted(pos)
        if 2 in row:
            hit += 1
            # a lower-id twin is always chosen before a higher-id twin
            assert row.index(2) < (row.index(9) if 9 in row else 99)
        if 14 in row:
            assert 2 in row and 9 in row
        if 9 in row:
            assert 2 in row
            # equal weights for equal logits
            assert wt[r, row.index(9)] == wt[r, row.index(2)]
    assert hit > 0


def test_weights_equal_full_softmax_then_renormalised(oracle_mod):
    """Top-k of the full 256-way softmax, renormalised, equals the k-way softmax."""
    w = W.BLOCK32
    x = u16(W.make_x(w))
    wr = u16(W.make_router(w))
    idx, wt, z, nf = oracle_mod.route(x, wr, w.block_offsets(), w.k, want_logits=True)
    for r in range(w.R):
        zz = z[r].astype(np.float64)
        p = np.exp(zz - zz.max())
        p /= p.sum()
        sel = p[idx[r]]
        ref = sel / sel.sum()
        assert np.allclose(wt[r], ref, rtol=2e-6, atol=0)
        s = np.float32(0)
        for v in wt[r]:
            s = np.float32(s + v)
        assert abs(float(s) - 1.0) <= w.k * 2.0 ** -23
        assert all(a >= b for a, b in zip(wt[r], wt[r][1:]))


def _softmax_hand_case(name):
    """A case of tests/golden/softmax_sums_hand.json as oracle inputs: one row with
    x one-hot at h = 0 and router rows whose element 0 is the wanted logit."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "softmax_sums_hand.json")
    with open(path) as f:
        fx = json.load(f)
    c = next(c for c in fx["cases"] if c["name"] == name)
    x = np.zeros((1, c["H"]), np.float32)
    x[0, 0] = 1.0
    wr = np.zeros((c["E"], c["H"]), np.float32)
    wr[:, 0] = c["other_logit"]
    for e, z in c["logits"].items():
        wr[int(e), 0] = z
    return c, fx["delta_arg"], bf16_bits(x), bf16_bits(wr)


def _hand_values(exprs, delta):
    """Values of the fixture's expressions in fp32 (1, delta, 1 - 2^-23, delta / (1 + 2^-23))."""
    one, d = np.float32(1.0), np.float32(delta)
    table = {"1": one, "delta": d, "1 - 2^-23": np.float32(1.0 - 2.0 ** -23),
             "delta / (1 + 2^-23)": np.float32(d / np.float32(1.0 + 2.0 ** -23))}
    return np.array([table[e] for e in exprs], np.float32)


def test_weight_sum_in_rank_order_hand_case(oracle_mod):
    """S = a_0 + ... + a_(k-1) summed in rank order, pinned at the bit level by a
    hand-worked row where rank order and id order give different fp32 sums
    (tests/golden/softmax_sums_hand.json, "S in rank order")."""
    c, darg, x, wr = _softmax_hand_case("S in rank order")
    delta = oracle_mod.exp_c(darg)
    # the derivation's premise: 1 + delta rounds to 1, 1 + 2 delta does not
    assert 2.0 ** -25 < delta < 2.0 ** -24
    assert np.float32(1.0) + np.float32(delta) == np.float32(1.0)
    assert np.float32(1.0) + np.float32(2 * delta) == np.float32(1.0 + 2.0 ** -23)
    idx, wt, _, _ = oracle_mod.route(x, wr, [0, 1], c["k"])
    assert idx[0].tolist() == c["topk_idx"]
    assert np.array_equal(wt[0].view(np.uint32), _hand_values(c["topk_w"], delta).view(np.uint32))


def test_prob_mass_denominator_in_lane_order_hand_case(oracle_mod):
    """The probability-mass reading: D = sum over all experts of exp_c(z_e - z_max)
    in the lane order (lane p sums experts p, p + 32, ...; then the xor
    butterfly), pinned at the bit level by a hand-worked row
    (tests/golden/softmax_sums_hand.json, "D in lane order")."""
    c, darg, x, wr = _softmax_hand_case("D in lane order")
    delta = oracle_mod.exp_c(darg)
    assert 2.0 ** -25 < delta < 2.0 ** -24
    idx, wt, _, _, p = oracle_mod.route(x, wr, [0, 1], c["k"], want_probs=True)
    assert idx[0].tolist() == c["topk_idx"]
    assert np.array_equal(wt[0].view(np.uint32), _hand_values(c["topk_w"], delta).view(np.uint32))
    assert p[0, 0].view(np.uint32) == 0x3F7FFFFE
    assert np.array_equal(p[0].view(np.uint32), _hand_values(c["topk_p"], delta).view(np.uint32))


def test_prob_mass_equals_full_softmax(oracle_mod):
    """p_j = the selected experts' probabilities under the softmax over all E
    experts (fp64 reference, within the fp32 summation and exp_c error), with
    p_j / w_j the same ratio S / D for every slot of a row."""
    w = W.BLOCK32
    x = u16(W.make_x(w))
    wr = u16(W.make_router(w))
    idx, wt, z, nf, p = oracle_mod.route(x, wr, w.block_offsets(), w.k, want_logits=True,
                                         want_probs=True)
    assert nf == 0
    for r in range(w.R):
        zz = z[r].astype(np.float64)
        full = np.exp(zz - zz.max())
        full /= full.sum()
        assert np.allclose(p[r], full[idx[r]], rtol=2e-5, atol=0)
        ratio = p[r].astype(np.float64) / wt[r].astype(np.float64)
        assert np.allclose(ratio, ratio[0], rtol=4e-7, atol=0)
        assert float(p[r].astype(np.float64).sum()) < 1.0
        assert all(a >= b for a, b in zip(p[r], p[r][1:]))


def test_prob_mass_same_ids_and_weights(oracle_mod):
    """Asking for the probability mass changes neither the ids nor the weights."""
    w = W.TINY
    T = W.make_tensors(w)
    a = oracle_mod.route(u16(T.x), u16(T.w_router), w.block_offsets(), w.k)
    b = oracle_mod.route(u16(T.x), u16(T.w_router), w.block_offsets(), w.k, want_probs=True)
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_nan_logits_rank_last(oracle_mod):
    w = W.TINY
    T = W.make_tensors(w)
    bias = np.zeros((1, w.E), np.float32)
    bias[0, 3] = np.nan
    bias[0, 5] = np.inf * -1
    idx, wt, z, nf = oracle_mod.route(u16(T.x), u16(T.w_router), [0, w.R], w.k, bias=bias,
                                      want_logits=True)
    assert nf == 2 * w.R
    assert not np.any(idx == 3) and not np.any(idx == 5)


# --------------------------------------------------------------------------- coreset

def _masses(idx, wt, r0, r1, E):
    Q = [0] * E
    touched = set()
    for r in range(r0, r1):
        for j in range(idx.shape[1]):
            e = int(idx[r, j])
            touched.add(e)
            Q[e] += int(Fraction(float(wt[r, j])) * (1 << 32))  # floor of an exact rational
    return Q, touched


def _theta(tau: float, T: int) -> int:
    return math.ceil(Fraction(float(np.float32(tau))) * T)


def _brute_min_size(Q, touched, theta):
    items = sorted(touched)
    for c in range(0, len(items) + 1):
        for sub in itertools.combinations(items, c):
            if sum(Q[e] for e in sub) >= theta:
                return c, sub
    raise AssertionError("no subset reaches theta")


def test_coreset_brute_force_tiny_config(oracle_mod):
    """Tiny config (16 experts): the coreset has the minimum size over all 2^16 subsets."""
    w = W.TINY
    T = W.make_tensors(w)
    idx, wt, _, _ = oracle_mod.route(u16(T.x), u16(T.w_router), w.block_offsets(), w.k)
    keep, cs, wr, ne, bad = oracle_mod.coreset(w.block_offsets(), idx, wt, w.E, w.tau)
    Q, touched = _masses(idx, wt, 0, w.R, w.E)
    theta = _theta(w.tau, sum(Q))
    # exhaustive over all subsets of the 16 experts (not only touched ones)
    best = None
    for mask in range(1 << w.E):
        m = sum(Q[e] for e in range(w.E) if mask >> e & 1)
        if m >= theta:
            c = bin(mask).count("1")
            best = c if best is None else min(best, c)
    core = [e for e in range(w.E) if keep[0, e // 32] >> (e % 32) & 1]
    assert cs[0] == len(core) == best
    assert sum(Q[e] for e in core) >= theta
    assert set(core) <= touched
    assert bad == 0 and ne[0] == 0


@pytest.mark.parametrize("seed", range(12))
def test_coreset_brute_force_random_tiny(oracle_mod, seed):
    """Random blocks over E <= 20 experts: minimal size, mass >= theta, greedy prefix,
    prefix of size c-1 below theta."""
    rng = np.random.default_rng(seed)
    E = int(rng.integers(4, 21))
    k = int(rng.integers(1, min(E, 6) + 1))
    nb = int(rng.integers(1, 4))
    rows = [int(rng.integers(1, 9)) for _ in range(nb)]
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    idx = np.zeros((R, k), np.int32)
    wt = np.zeros((R, k), np.float32)
    for r in range(R):
        idx[r] = rng.choice(E, size=k, replace=False)
        a = np.sort(rng.random(k).astype(np.float32))[::-1] + np.float32(0.01)
        wt[r] = (a / a.sum()).astype(np.float32)
    tau = float(np.float32(rng.choice([0.5, 0.75, 0.9, 0.95, 0.999])))
    keep, cs, wr, ne, bad = oracle_mod.coreset(off, idx, wt, E, tau)
    for b in range(nb):
        Q, touched = _masses(idx, wt, off[b], off[b + 1], E)
        theta = _theta(tau, sum(Q))
        cmin, _ = _brute_min_size(Q, touched, theta)
        core = [e for e in range(E) if keep[b, e // 32] >> (e % 32) & 1]
        assert cs[b] == len(core) == cmin
        assert sum(Q[e] for e in core) >= theta
        order = sorted(touched, key=lambda e: (-Q[e], e))
        assert core == sorted(order[:cmin])
        assert sum(Q[e] for e in order[:cmin - 1]) < theta
        # renormalisation: surviving weights of each row sum to 1
        for r in range(off[b], off[b + 1]):
            surv = [j for j in range(k) if idx[r, j] in core]
            if not surv:
                assert np.all(wr[r] == 0)
                continue
            s = np.float32(0)
            for j in surv:
                s = np.float32(s + wt[r, j])
            for j in range(k):
                expect = np.float32(wt[r, j] / s) if j in surv else np.float32(0)
                assert wr[r, j] == expect
            assert abs(float(wr[r].astype(np.float64).sum()) - 1.0) <= k * 2.0 ** -23


def _random_tiny_blocks(rng):
    E = int(rng.integers(4, 21))
    k = int(rng.integers(1, min(E, 6) + 1))
    nb = int(rng.integers(1, 4))
    rows = [int(rng.integers(1, 9)) for _ in range(nb)]
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    idx = np.zeros((R, k), np.int32)
    wt = np.zeros((R, k), np.float32)
    for r in range(R):
        idx[r] = rng.choice(E, size=k, replace=False)
        a = np.sort(rng.random(k).astype(np.float32))[::-1] + np.float32(0.01)
        wt[r] = (a / a.sum()).astype(np.float32)
    return E, k, nb, off, idx, wt


@pytest.mark.parametrize("seed", range(8))
def test_coreset_budget_brute_force_random_tiny(oracle_mod, seed):
    """Expert budget B: the kept set has size min(c, B) (c = the minimal size
    reaching theta, by brute force) and the largest mass of any set of that
    size (brute force), ties to lower ids; rows renormalised over it."""
    rng = np.random.default_rng(100 + seed)
    E, k, nb, off, idx, wt = _random_tiny_blocks(rng)
    tau = float(np.float32(rng.choice([0.5, 0.75, 0.9, 0.999, 1.0])))
    B = int(rng.integers(1, E + 1))
    keep, cs, wr, ne, bad = oracle_mod.coreset(off, idx, wt, E, tau, max_experts=B)
    for b in range(nb):
        Q, touched = _masses(idx, wt, off[b], off[b + 1], E)
        items = sorted(touched)
        if tau < 1.0:
            cmin, _ = _brute_min_size(Q, touched, _theta(tau, sum(Q)))
        else:
            cmin = len(items)
        size = min(cmin, B)
        best = max(sum(Q[e] for e in sub) for sub in itertools.combinations(items, size))
        core = [e for e in range(E) if keep[b, e // 32] >> (e % 32) & 1]
        assert cs[b] == len(core) == size
        assert sum(Q[e] for e in core) == best
        # among the sets of that mass, the one preferring lower ids at equal mass
        order = sorted(touched, key=lambda e: (-Q[e], e))
        assert core == sorted(order[:size])
        renorm = tau < 1.0 or size < len(items)
        for r in range(off[b], off[b + 1]):
            if not renorm:
                assert np.array_equal(wr[r].view(np.uint32), wt[r].view(np.uint32))
                continue
            surv = [j for j in range(k) if idx[r, j] in core]
            s = np.float32(0)
            for j in surv:
                s = np.float32(s + wt[r, j])
            for j in range(k):
                expect = np.float32(wt[r, j] / s) if (j in surv and s > 0) else np.float32(0)
                assert wr[r, j] == expect


@pytest.mark.parametrize("seed", range(6))
def test_coreset_prob_mass_brute_force_random_tiny(oracle_mod, seed):
    """Masses given apart from the weights (the probability-mass reading): each row's
    masses are its weights times its own factor in (0, 1), so the rows carry unequal
    mass.  The kept set is the minimal one reaching ceil(tau * T) of those masses
    (brute force), the greedy prefix under (mass desc, id asc); the rows are still
    renormalised from their weights."""
    rng = np.random.default_rng(200 + seed)
    E, k, nb, off, idx, wt = _random_tiny_blocks(rng)
    R = idx.shape[0]
    scale = (rng.random(R).astype(np.float32) * np.float32(0.9) + np.float32(0.05))
    mass = (wt * scale[:, None]).astype(np.float32)
    tau = float(np.float32(rng.choice([0.5, 0.75, 0.9, 0.95])))
    B = int(rng.integers(0, E + 1)) if seed % 2 else 0
    keep, cs, wr, ne, bad = oracle_mod.coreset(off, idx, wt, E, tau, max_experts=B, mass=mass)
    for b in range(nb):
        Q, touched = _masses(idx, mass, off[b], off[b + 1], E)
        cmin, _ = _brute_min_size(Q, touched, _theta(tau, sum(Q)))
        size = min(cmin, B) if B > 0 else cmin
        order = sorted(touched, key=lambda e: (-Q[e], e))
        core = [e for e in range(E) if keep[b, e // 32] >> (e % 32) & 1]
        assert cs[b] == len(core) == size
        assert core == sorted(order[:size])
        for r in range(off[b], off[b + 1]):
            surv = [j for j in range(k) if idx[r, j] in core]
            s = np.float32(0)
            for j in surv:
                s = np.float32(s + wt[r, j])
            for j in range(k):
                expect = np.float32(wt[r, j] / s) if (j in surv and s > 0) else np.float32(0)
                assert wr[r, j] == expect


def test_coreset_prob_mass_changes_membership(oracle_mod):
    """Unequal row masses change some block's coreset against the weight reading
    (so the pin above checks the mass input and not only the weights)."""
    changed = 0
    for seed in range(200, 220):
        rng = np.random.default_rng(seed)
        E, k, nb, off, idx, wt = _random_tiny_blocks(rng)
        scale = (rng.random(idx.shape[0]).astype(np.float32) * np.float32(0.9) + np.float32(0.05))
        mass = (wt * scale[:, None]).astype(np.float32)
        a = oracle_mod.coreset(off, idx, wt, E, 0.75, mass=mass)[0]
        b = oracle_mod.coreset(off, idx, wt, E, 0.75)[0]
        changed += not np.array_equal(a, b)
    assert changed >= 3


def test_coreset_prob_mass_on_full_shape_block(oracle_mod):
    """The 32-row block under the probability mass: invariants of the cut (mass >=
    theta, the prefix one shorter below it) on the masses q = trunc(p * 2^32)."""
    w = W.BLOCK32
    x = u16(W.make_x(w))
    wrt = u16(W.make_router(w))
    idx, wt, _, _, p = oracle_mod.route(x, wrt, w.block_offsets(), w.k, want_probs=True)
    keep, cs, wr, ne, bad = oracle_mod.coreset(w.block_offsets(), idx, wt, w.E, w.tau, mass=p)
    Q, touched = _masses(idx, p, 0, w.R, w.E)
    theta = _theta(w.tau, sum(Q))
    core = [e for e in range(w.E) if keep[0, e // 32] >> (e % 32) & 1]
    order = sorted(touched, key=lambda e: (-Q[e], e))
    assert core == sorted(order[:cs[0]])
    assert sum(Q[e] for e in core) >= theta > sum(Q[e] for e in order[:cs[0] - 1])
    assert bad == 0


def test_coreset_budget_hand_example(oracle_mod):
    """Hand-worked block (masses Q0 = 2^32 > Q1 = Q2 = 2^31, see below): budget 1
    keeps expert 0 only; with tau = 1 and budget 2 experts {0, 1} (equal masses
    go to the lower id) and the rows are renormalised; budget 0 or 3 changes
    nothing."""
    idx = np.array([[0, 1], [0, 2]], np.int32)
    wt = np.full((2, 2), 0.5, np.float32)
    off = [0, 2]
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 0.75, max_experts=1)
    assert cs[0] == 1 and keep[0, 0] == 0b001
    assert np.array_equal(wr, np.array([[1, 0], [1, 0]], np.float32))
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 1.0, max_experts=2)
    assert cs[0] == 2 and keep[0, 0] == 0b011
    assert np.array_equal(wr, np.array([[0.5, 0.5], [1, 0]], np.float32))
    for B in (0, 3):
        keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 1.0, max_experts=B)
        assert cs[0] == 3 and keep[0, 0] == 0b111 and np.array_equal(wr, wt)


def test_coreset_threshold_hand_example(oracle_mod):
    """Hand-worked block: 2 rows, k = 2, weights 0.5 (q = 2^31 each).
    Row 0 -> experts {0, 1}, row 1 -> {0, 2}: Q0 = 2^32, Q1 = Q2 = 2^31, T = 2^33.
    tau = 0.5 -> theta = 2^32 -> coreset {0}; tau = 0.75f -> theta = 3*2^31 -> {0, 1}
    (tie Q1 = Q2 goes to the lower id); w' of row 0 = [1, 0] / [2/3?]: row 0 keeps
    both experts under tau 0.75 (w' = w / 1.0 = 0.5 each), row 1 keeps only expert 0
    (w' = 0.5 / 0.5 = 1)."""
    off = [0, 2]
    idx = np.array([[0, 1], [0, 2]], np.int32)
    wt = np.full((2, 2), 0.5, np.float32)
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 0.5)
    assert cs[0] == 1 and keep[0, 0] == 0b001
    assert wr.tolist() == [[1.0, 0.0], [1.0, 0.0]]
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 0.75)
    assert cs[0] == 2 and keep[0, 0] == 0b011
    assert wr.tolist() == [[0.5, 0.5], [1.0, 0.0]]
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 3, 1.0)
    assert cs[0] == 3 and keep[0, 0] == 0b111
    assert wr.tolist() == wt.tolist()


def test_coreset_threshold_is_ceiling(oracle_mod):
    """One row, k = 3, w = (0.375, 0.375, 2^-32): Q = (3*2^29, 3*2^29, 1), T odd.
    tau = 0.5: tau*T = 3*2^29 + 0.5, so theta = 3*2^29 + 1 and the first expert alone
    (mass 3*2^29) falls short by one unit: the coreset is {0, 1}."""
    idx = np.array([[0, 1, 2]], np.int32)
    wt = np.array([[0.375, 0.375, 2.0 ** -32]], np.float32)
    keep, cs, wr, ne, _ = oracle_mod.coreset([0, 1], idx, wt, 3, 0.5)
    assert cs[0] == 2 and keep[0, 0] == 0b011
    assert wr.tolist() == [[0.5, 0.5, 0.0]]


def test_coreset_empty_row_counted(oracle_mod):
    """A row whose experts all fall outside the coreset keeps only the shared expert."""
    off = [0, 3]
    idx = np.array([[0], [0], [1]], np.int32)
    wt = np.ones((3, 1), np.float32)
    keep, cs, wr, ne, _ = oracle_mod.coreset(off, idx, wt, 2, 0.6)
    assert cs[0] == 1 and ne[0] == 1
    assert wr[:, 0].tolist() == [1.0, 1.0, 0.0]


def test_coreset_disabled_is_plain_topk(oracle_mod):
    """tau >= 1: every touched expert kept and w' == w bit for bit."""
    w = W.TINY
    T = W.make_tensors(w)
    idx, wt, _, _ = oracle_mod.route(u16(T.x), u16(T.w_router), w.block_offsets(), w.k)
    for tau in (1.0, 1.5, float("inf")):
        keep, cs, wr, ne, _ = oracle_mod.coreset(w.block_offsets(), idx, wt, w.E, tau)
        touched = sorted(set(idx.reshape(-1).tolist()))
        core = [e for e in range(w.E) if keep[0, e // 32] >> (e % 32) & 1]
        assert core == touched and cs[0] == len(touched)
        assert np.array_equal(wr.view(np.uint32), wt.view(np.uint32))


def test_coreset_rejects_bad_tau(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.coreset([0, 1], np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), 1,
                           0.0)
    with pytest.raises(ValueError):
        oracle_mod.coreset([0, 1], np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), 1,
                           float("nan"))


def test_coreset_multiblock_is_blockwise(oracle_mod):
    """Each block's coreset depends only on its own rows."""
    w = W.blocks2048(8, 0.9)
    x = u16(W.make_x(w, rows=64))
    wr_ = u16(W.make_router(w))
    off = list(range(0, 65, 8))
    idx, wt, _, _ = oracle_mod.route(x, wr_, off, 8)
    keep, cs, wrn, ne, _ = oracle_mod.coreset(off, idx, wt, 256, 0.9)
    for b in range(8):
        k1, c1, w1, _, _ = oracle_mod.coreset([0, 8], idx[8 * b:8 * b + 8], wt[8 * b:8 * b + 8],
                                             256, 0.9)
        assert np.array_equal(k1[0], keep[b]) and c1[0] == cs[b]
        assert np.array_equal(w1, wrn[8 * b:8 * b + 8])


# --------------------------------------------------------------------------- FFN

def _f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def _swiglu_np(xr, wg, wu, wd):
    g = _f64(wg) @ xr
    u = _f64(wu) @ xr
    h = g / (1.0 + np.exp(-g)) * u
    return _f64(wd) @ h


def test_expert_ffn_hand_value(oracle_mod):
    """H = 2, I = 1: x = (1, 2), Wg = (0.5, 0.25) -> g = 1; Wu = (1, -1) -> u = -1;
    h = silu(1) * -1 = -1/(1+e^-1); Wd = (2, -4)^T -> out = (2h, -4h)."""
    x = bf16_bits([1.0, 2.0])
    wg = bf16_bits([[0.5, 0.25]])
    wu = bf16_bits([[1.0, -1.0]])
    wd = bf16_bits([[2.0], [-4.0]])
    out = oracle_mod.expert_ffn(x, wg, wu, wd)
    h = -1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(out, [2 * h, -4 * h], rtol=1e-15, atol=0)


def test_expert_ffn_matches_dense_fp64(oracle_mod):
    w = W.TINY
    T = W.make_tensors(w)
    x = u16(T.x)
    wg, wu, wd = u16(T.w_gate), u16(T.w_up), u16(T.w_down)
    for r in (0, 7, 31):
        for e in (0, 5, 15):
            got = oracle_mod.expert_ffn(x[r], wg[e], wu[e], wd[e])
            ref = _swiglu_np(_f64(x[r]), wg[e], wu[e], wd[e])
            assert np.allclose(got, ref, rtol=1e-10, atol=1e-13)


def _tiny_setup(oracle_mod, tau):
    w = W.TINY
    T = W.make_tensors(w)
    x = u16(T.x)
    idx, wt, _, _ = oracle_mod.route(x, u16(T.w_router), w.block_offsets(), w.k)
    keep, cs, wr, ne, _ = oracle_mod.coreset(w.block_offsets(), idx, wt, w.E, tau)
    experts = {e: (u16(T.w_gate[e]), u16(T.w_up[e]), u16(T.w_down[e])) for e in range(w.E)}
    shared = (u16(T.ws_gate), u16(T.ws_up), u16(T.ws_down))
    return w, T, x, idx, wt, keep, wr, experts, shared


def test_forward_matches_dense_moe_fp64(oracle_mod):
    """y = S(x) + sum over surviving pairs w' E_e(x), evaluated densely in numpy."""
    w, T, x, idx, wt, keep, wr, experts, shared = _tiny_setup(oracle_mod, 0.9)
    y = oracle_mod.forward(x, w.block_offsets(), idx, wr, keep, experts, shared, w.E)
    mask = oracle_mod.keep_mask(keep, w.E)
    for r in range(w.R):
        xr = _f64(x[r])
        ref = _swiglu_np(xr, *shared)
        for j in range(w.k):
            e = idx[r, j]
            if mask[0, e]:
                ref = ref + float(wr[r, j]) * _swiglu_np(xr, *experts[e])
        assert np.allclose(y[r], ref, rtol=1e-10, atol=1e-12)


def test_forward_coreset_disabled_equals_plain_topk_moe(oracle_mod):
    """tau >= 1: the coreset forward is the plain top-k MoE with the router weights."""
    w, T, x, idx, wt, keep, wr, experts, shared = _tiny_setup(oracle_mod, 1.0)
    y = oracle_mod.forward(x, w.block_offsets(), idx, wr, keep, experts, shared, w.E)
    for r in range(w.R):
        xr = _f64(x[r])
        ref = _swiglu_np(xr, *shared)
        for j in range(w.k):
            ref = ref + float(wt[r, j]) * _swiglu_np(xr, *experts[idx[r, j]])
        assert np.allclose(y[r], ref, rtol=1e-10, atol=1e-12)


def test_forward_linear_in_weights_and_row_subset(oracle_mod):
    w, T, x, idx, wt, keep, wr, experts, shared = _tiny_setup(oracle_mod, 0.9)
    off = w.block_offsets()
    y1 = oracle_mod.forward(x, off, idx, wr, keep, experts, shared, w.E)
    y2 = oracle_mod.forward(x, off, idx, wr * np.float32(2), keep, experts, shared, w.E)
    y0 = oracle_mod.forward(x, off, idx, wr * np.float32(0), keep, experts, shared, w.E)
    assert np.allclose(y2 - y0, 2 * (y1 - y0), rtol=1e-9, atol=1e-12)
    ys = oracle_mod.forward(x, off, idx, wr, keep, experts, shared, w.E, rows=[3, 17])
    assert np.array_equal(ys[[3, 17]], y1[[3, 17]])
    assert np.all(ys[[0, 1, 2]] == 0)


def test_forward_live_rows(oracle_mod):
    """Live-row pass: each live row equals the dense numpy MoE of that row, each dead
    row keeps its cached value bit for bit; all live = the full forward, none live =
    the cache."""
    w, T, x, idx, wt, keep, wr, experts, shared = _tiny_setup(oracle_mod, 0.9)
    off = w.block_offsets()
    cached = np.random.default_rng(5).standard_normal((w.R, w.H))
    live = W.live_rows(w.R, 0.4, seed=11).numpy()
    assert 0 < live.sum() < w.R
    y = oracle_mod.forward_live(x, off, idx, wr, keep, experts, shared, w.E, live, cached)
    mask = oracle_mod.keep_mask(keep, w.E)
    for r in range(w.R):
        if not live[r]:
            assert np.array_equal(y[r], cached[r])
            continue
        xr = _f64(x[r])
        ref = _swiglu_np(xr, *shared)
        for j in range(w.k):
            if mask[0, idx[r, j]]:
                ref = ref + float(wr[r, j]) * _swiglu_np(xr, *experts[idx[r, j]])
        assert np.allclose(y[r], ref, rtol=1e-10, atol=1e-12)
    full = oracle_mod.forward(x, off, idx, wr, keep, experts, shared, w.E)
    ones = np.ones(w.R, np.uint8)
    assert np.array_equal(
        oracle_mod.forward_live(x, off, idx, wr, keep, experts, shared, w.E, ones, cached), full)
    zeros = np.zeros(w.R, np.uint8)
    assert np.array_equal(
        oracle_mod.forward_live(x, off, idx, wr, keep, experts, shared, w.E, zeros, cached),
        cached)


def test_forward_missing_expert_is_an_error(oracle_mod):
    w, T, x, idx, wt, keep, wr, experts, shared = _tiny_setup(oracle_mod, 0.9)
    used = oracle_mod.surviving_experts(idx, keep, w.block_offsets(), w.E)
    partial = {e: experts[e] for e in used[1:]}
    with pytest.raises(KeyError):
        oracle_mod.forward(x, w.block_offsets(), idx, wr, keep, partial, shared, w.E)
    only = {e: experts[e] for e in used}
    y = oracle_mod.forward(x, w.block_offsets(), idx, wr, keep, only, shared, w.E)
    assert np.isfinite(y).all()


# --------------------------------------------------------------------------- quantised experts

def _quant_hand_cases():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "quant_hand.json")
    with open(path) as f:
        return json.load(f)["cases"]


def test_dequant_hand_cases(oracle_mod):
    """Quantised weights back to bf16 against the hand-worked blocks of
    tests/golden/quant_hand.json: products, a rounding, a tie to even, the nibble
    order and sign, and the block-major scale layout."""
    for c in _quant_hand_cases():
        rows, K, bits = c["rows"], c["K"], c["bits"]
        d = bf16_bits(np.array(c["scales_block_major"], np.float32).reshape(-1)).reshape(K // 32, rows)
        if bits == 8:
            q = np.zeros((rows, K), np.int8)
            for r, cols in c["q"].items():
                for k, v in cols.items():
                    q[int(r), int(k)] = v
        else:
            q = np.zeros((rows, K // 2), np.uint8)
            for r, cols in c["bytes"].items():
                for k, v in cols.items():
                    q[int(r), int(k)] = int(v, 16)
        want = np.zeros((rows, K), np.float32)
        for r, cols in c["w"].items():
            for k, v in cols.items():
                want[int(r), int(k)] = v
        got = oracle_mod.dequant(q, d, bits)
        assert np.array_equal(got, bf16_bits(want)), c["name"]


@pytest.mark.parametrize("bits", [8, 4])
def test_dequant_round_trip_of_the_synthetic_quantiser(oracle_mod, bits):
    """The synthetic quantiser followed by the oracle's dequantisation: every weight
    within half a step (d / 2) plus its bf16 rounding of the original, and the
    all-zero q of a zero block gives +0."""
    w = W.TINY
    T = W.make_tensors(w)
    q, d = W.quantize_rows(T.w_gate[:2], bits)
    qs = W.pack_int4(q) if bits == 4 else q
    dq = oracle_mod.dequant(qs.numpy(), u16(W.scales_k_major(d)), bits)
    back = torch.from_numpy(dq.view(np.int16)).view(torch.bfloat16).float()
    step = d.float().repeat_interleave(32, dim=-1)
    orig = T.w_gate[:2].float()
    assert torch.all((back - orig).abs() <= step / 2 + orig.abs() * 2.0 ** -8 + 1e-30)
    assert not torch.equal(back, orig)   # it is a real quantisation
