"""Pins for the CPU oracle: each check ties it to something other than itself
(IEEE format definitions, exact rational arithmetic, brute force on tiny
inputs, closed forms, invariants, textbook values, a hand-worked trace)."""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
from scipy.special import erf as sp_erf

import oracle
from workload import TINY, Shape, gen_hidden, gen_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers (test-side, independent)

def np_fp16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def np_bf16(bits):
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns widen to NaN
        return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense_dequant(q, sb, group=64):
    """Materialise an int4 affine matrix with numpy bit operations."""
    q = np.asarray(q, dtype=np.uint8)
    rows, half = q.shape
    vals = np.empty((rows, 2 * half), dtype=np.float64)
    vals[:, 0::2] = q & 0x0F
    vals[:, 1::2] = q >> 4
    sbf = np_fp16(oracle.as_bits(sb)).reshape(rows, -1, 2)
    s = np.repeat(sbf[:, :, 0], group, axis=1)
    b = np.repeat(sbf[:, :, 1], group, axis=1)
    return s * vals + b


def gelu_ref(x):
    return 0.5 * x * (1.0 + sp_erf(x / np.sqrt(2.0)))


def dense_ffn(w, x, group=64):
    g = dense_dequant(w["gate_q"], w["gate_sb"], group) @ x
    u = dense_dequant(w["up_q"], w["up_sb"], group) @ x
    return dense_dequant(w["down_q"], w["down_sb"], group) @ (gelu_ref(g) * u)


def expert_slice(ex, e):
    return {k: v[e] for k, v in ex.items()}


# ----------------------------------------------------------------- 16-bit float formats

def test_fp16_decoding_matches_ieee_binary16_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = np_fp16(bits)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decoding_matches_float32_upper_half_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = np_bf16(bits)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])


def _nearest_bf16_bruteforce(v):
    """Nearest bf16 to v by scanning neighbours of a float32 guess; ties to even."""
    guess = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
    best = None
    for b in range(max(0, guess - 2), min(0xFFFF, guess + 3)):
        if (b & 0x7F80) == 0x7F80:
            continue
        val = float(np_bf16([b])[0])
        if math.copysign(1.0, val) != math.copysign(1.0, v) and val != 0.0:
            continue
        dist = abs(val - v)
        key = (dist, b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_bf16_rounding_is_nearest_ties_to_even():
    one = 0x3F80
    assert oracle.double_to_bf16(1.0) == one
    assert oracle.double_to_bf16(1.0 + 2 ** -8) == one            # midpoint, even stays
    assert oracle.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82      # midpoint, rounds to even
    assert oracle.double_to_bf16(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.double_to_bf16(-2.5) == 0xC020
    assert oracle.double_to_bf16(3.3895313892515355e38) == 0x7F7F  # largest finite bf16
    assert oracle.double_to_bf16(4e38) == 0x7F80
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                           rng.standard_normal(500) * 1e-39])
    for v in vals:
        v = float(v)
        assert oracle.double_to_bf16(v) == _nearest_bf16_bruteforce(v), v


# ----------------------------------------------------------------- router

def _fraction_logits(w_bits, x_bits, bias=None):
    W = [[Fraction(float(v)) for v in row] for row in np_fp16(w_bits)]
    X = [Fraction(float(v)) for v in np_bf16(x_bits)]
    two40 = Fraction(2) ** 40
    out = []
    for e, row in enumerate(W):
        acc = sum(round(wi * xi * two40) for wi, xi in zip(row, X))
        if bias is not None:
            acc += round(Fraction(float(bias[e])) * two40)
        out.append(acc)
    return out


def test_router_fixed_point_matches_exact_rationals():
    rng = np.random.default_rng(2)
    for trial in range(4):
        E, d = 6, 64
        w = torch.from_numpy(rng.standard_normal((E, d)) * 0.02).to(torch.float16)
        x = torch.from_numpy(rng.standard_normal(d) * (10.0 ** (trial - 2))).to(torch.bfloat16)
        bias = rng.standard_normal(E).astype(np.float32) if trial % 2 else None
        got, st = oracle.router_logits(w, x, bias)
        assert st == 0
        ref = _fraction_logits(oracle.as_bits(w), oracle.as_bits(x), bias)
        assert [int(v) for v in got] == ref


def test_router_domain_error_on_huge_products():
    w = torch.full((2, 64), 1000.0, dtype=torch.float16)
    x = torch.full((64,), 100.0, dtype=torch.bfloat16)
    _, st = oracle.router_logits(w, x)
    assert st != 0


def test_topk_equals_full_stable_sort_with_ties():
    rng = np.random.default_rng(3)
    for _ in range(300):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-3, 4, size=E).astype(np.int64)   # many ties
        ref = sorted(range(E), key=lambda e: (-lg[e], e))[:k]
        assert list(oracle.topk(lg, k)) == ref


def test_gates_invariants_and_closed_forms():
    rng = np.random.default_rng(4)
    lg = rng.integers(-2 ** 42, 2 ** 42, size=16).astype(np.int64)
    ids = oracle.topk(lg, 5)
    g = oracle.gates(lg, ids)
    assert abs(g.sum() - 1.0) < 1e-15
    assert np.all(np.diff(g) <= 0)                      # ranked order gives non-increasing gates
    # softmax over all E, then renormalised over the picked k, is the same value
    z = np.exp((lg - lg.max()) / 2.0 ** 40)
    sm = z / z.sum()
    ref = sm[ids] / sm[ids].sum()
    assert np.allclose(g, ref, rtol=1e-13, atol=0)
    assert oracle.gates(lg, ids[:1])[0] == 1.0          # k = 1 gives weight 1
    eq = np.zeros(8, dtype=np.int64)
    assert np.all(oracle.gates(eq, np.arange(4, dtype=np.int32)) == 0.25)
    # logits one ln(2) apart: gates 2/3 and 1/3
    delta = int(round(math.log(2.0) * 2 ** 40))
    two = np.array([delta, 0], dtype=np.int64)
    g2 = oracle.gates(two, np.array([0, 1], dtype=np.int32))
    assert abs(g2[0] - 2 / 3) < 1e-12 and abs(g2[1] - 1 / 3) < 1e-12


# ----------------------------------------------------------------- int4 affine FFN

def test_gelu_textbook_values():
    # Phi(1) and Phi(2), standard normal CDF
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu(2.0) - 2 * 0.9772498680518208) < 1e-15
    assert oracle.gelu(0.0) == 0.0
    for x in (-3.0, -0.7, 0.3, 1.9, 5.0):
        assert abs((oracle.gelu(x) - oracle.gelu(-x)) - x) < 1e-15
        assert abs(oracle.gelu(x, 1) - oracle.gelu(x, 0)) < 1e-3    # tanh form approximates erf form


def test_gelu_tanh_form_against_decimal_values():
    # the tanh variant against the formula evaluated in 50-digit decimal
    # arithmetic by tests/golden/make_gelu_tanh.py (no float library involved):
    # a wrong coefficient (0.044715, sqrt(2/pi)) or a dropped term moves these
    # values by far more than the tolerance
    import json
    with open(os.path.join(os.path.dirname(__file__), "golden", "gelu_tanh.json")) as fh:
        g = json.load(fh)
    assert len(g["values"]) >= 10
    for x, v in g["values"]:
        got, ref = oracle.gelu(float(x), 1), float(v)
        assert abs(got - ref) <= 1e-15 + 1e-15 * abs(ref), (x, got, ref)


def test_matvec_matches_materialised_dense_matrix():
    sh = Shape(d=192, f=64, f_shared=64, n_experts=2, top_k=1)
    L = gen_layer(sh, seed=11, layer=0)
    x = np.random.default_rng(5).standard_normal(192)
    for name in ("gate", "up"):
        q, sb = L["shared"][name + "_q"], L["shared"][name + "_sb"]
        ref = dense_dequant(q.numpy(), sb) @ x
        got = oracle.matvec(q, sb, x)
        assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_int4_special_cases_closed_forms():
    rows, cols, grp = 4, 128, 64
    x = np.random.default_rng(6).standard_normal(cols)
    # all q = 0: W = bias per group, y = sum_g b_g * sum_{c in g} x_c
    q0 = np.zeros((rows, cols // 2), dtype=np.uint8)
    b = np.array([[0.5, -0.25], [1.0, 2.0], [0.0, -1.5], [0.125, 0.0]], dtype=np.float16)
    sb = np.stack([np.full_like(b, 0.75), b], -1).astype(np.float16).view(np.uint16)
    got = oracle.matvec(q0, np.ascontiguousarray(sb), x)
    X = x.reshape(2, 64).sum(1)
    assert np.allclose(got, b.astype(np.float64) @ X, rtol=1e-14, atol=1e-14)
    # scale = 0, bias = c: y = c * sum(x) regardless of q
    q = np.random.default_rng(7).integers(0, 256, (rows, cols // 2)).astype(np.uint8)
    sbc = np.zeros((rows, 2, 2), dtype=np.float16)
    sbc[..., 1] = 0.375
    got = oracle.matvec(q, np.ascontiguousarray(sbc.view(np.uint16)), x)
    assert np.allclose(got, 0.375 * x.sum(), rtol=1e-14, atol=1e-14)
    # q = 15 everywhere with s = 1, b = 0: y = 15 * sum(x)
    q15 = np.full((rows, cols // 2), 0xFF, dtype=np.uint8)
    sb1 = np.zeros((rows, 2, 2), dtype=np.float16)
    sb1[..., 0] = 1.0
    got = oracle.matvec(q15, np.ascontiguousarray(sb1.view(np.uint16)), x)
    assert np.allclose(got, 15 * x.sum(), rtol=1e-14, atol=1e-13)
    # nibble order: element 2m is the low nibble of byte m
    qa = np.zeros((1, cols // 2), dtype=np.uint8)
    qa[0, 3] = 0x0A          # element 6 = 10, element 7 = 0
    qa[0, 40] = 0x50         # element 80 = 0, element 81 = 5
    sb1 = np.zeros((1, 2, 2), dtype=np.float16)
    sb1[..., 0] = 1.0
    e = np.zeros(cols)
    e[6], e[81] = 1.0, 100.0
    assert oracle.matvec(qa, np.ascontiguousarray(sb1.view(np.uint16)), e)[0] == 10.0 + 500.0


def test_expert_ffn_matches_dense_numpy():
    L = gen_layer(TINY, seed=12, layer=0)
    x = np_bf16(oracle.as_bits(gen_hidden(1, TINY.d, seed=12)[0]))
    for e in range(TINY.n_experts):
        w = expert_slice(L["experts"], e)
        assert np.allclose(oracle.expert_ffn(w, x), dense_ffn(w, x), rtol=1e-11, atol=1e-12)
    assert np.allclose(oracle.expert_ffn(L["shared"], x), dense_ffn(L["shared"], x), rtol=1e-11,
                       atol=1e-12)


def test_zero_gate_projection_gives_zero_output():
    L = gen_layer(TINY, seed=13, layer=0)
    w = {k: v.clone() for k, v in L["shared"].items()}
    w["gate_q"].zero_()
    w["gate_sb"].zero_()
    x = np_bf16(oracle.as_bits(gen_hidden(1, TINY.d, seed=13)[0]))
    assert np.all(oracle.expert_ffn(w, x) == 0.0)


def test_tiny_layer_matches_dense_brute_force():
    L = gen_layer(TINY, seed=0, layer=0)
    lay = oracle.Layer(L, TINY.top_k)
    H = gen_hidden(8, TINY.d, seed=0)
    for t in range(8):
        xb = oracle.as_bits(H[t])
        ids, g, lg, y, st = lay.forward(xb)
        assert st == 0
        ref_lg = _fraction_logits(oracle.as_bits(L["router_w"]), xb)
        assert [int(v) for v in lg] == ref_lg
        order = sorted(range(TINY.n_experts), key=lambda e: (-ref_lg[e], e))[:TINY.top_k]
        assert list(ids) == order
        x = np_bf16(xb)
        ref = dense_ffn(L["shared"], x)
        for j, e in enumerate(order):
            ref = ref + g[j] * dense_ffn(expert_slice(L["experts"], e), x)
        assert np.allclose(y, ref, rtol=1e-11, atol=1e-12)


def test_dense_equivalence_invariant():
    """Router weights 0, no bias, k = E: every logit ties at 0, ids = 0..E-1,
    gates 1/E, so y = FFN_shared(x) + mean_e FFN_e(x)."""
    sh = TINY
    L = gen_layer(sh, seed=14, layer=0)
    L["router_w"] = torch.zeros_like(L["router_w"])
    lay = oracle.Layer(L, top_k=sh.n_experts)
    xb = oracle.as_bits(gen_hidden(1, sh.d, seed=14)[0])
    ids, g, lg, y, st = lay.forward(xb)
    assert list(ids) == list(range(sh.n_experts))
    assert np.all(g == 1.0 / sh.n_experts)
    x = np_bf16(xb)
    mean = sum(dense_ffn(expert_slice(L["experts"], e), x) for e in range(sh.n_experts)) / sh.n_experts
    assert np.allclose(y, dense_ffn(L["shared"], x) + mean, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------- residual stream

def test_rmsnorm_closed_forms():
    one = oracle.double_to_bf16(1.0)
    h = np.full(64, one, dtype=np.uint16)
    assert np.all(oracle.rmsnorm_bf16(h, eps=1e-6) == one)   # 1/sqrt(1+1e-6) rounds to 1
    rng = np.random.default_rng(8)
    hb = oracle.as_bits(torch.from_numpy(rng.standard_normal(256)).to(torch.bfloat16))
    h2 = oracle.as_bits(torch.from_numpy(2.0 * np_bf16(hb)).to(torch.bfloat16))   # exact doubling
    assert np.array_equal(oracle.rmsnorm_bf16(hb, eps=0.0), oracle.rmsnorm_bf16(h2, eps=0.0))
    x = np_bf16(oracle.rmsnorm_bf16(hb, eps=1e-6))
    ref = np_bf16(hb) / np.sqrt(np.mean(np_bf16(hb) ** 2) + 1e-6)
    assert np.all(np.abs(x - ref) <= np.abs(ref) * 2.0 ** -8)


def test_residual_rounds_to_nearest_bf16():
    rng = np.random.default_rng(9)
    hb = oracle.as_bits(torch.from_numpy(rng.standard_normal(200) * 4).to(torch.bfloat16))
    y = rng.standard_normal(200)
    out = oracle.residual_bf16(hb, y)
    for i in range(200):
        assert out[i] == _nearest_bf16_bruteforce(float(np_bf16([hb[i]])[0] + y[i]))


# ----------------------------------------------------------------- LRU slot cache

def test_lru_hand_worked_trace():
    with open(os.path.join(GOLDEN, "lru_hand_trace.json")) as fh:
        g = json.load(fh)
    lru = oracle.LRU(g["n_slots"])
    hits = misses = 0
    for st in g["steps"]:
        hit, slot, ev = lru.step(st["ids"], st["t"])
        assert list(hit) == st["hit"]
        assert list(slot) == st["slot"]
        assert list(ev) == st["evicted"]
        hits += int(hit.sum())
        misses += int(len(hit) - hit.sum())
    assert hits == g["total_hits"] and misses == g["total_misses"]
    assert list(lru.expert_of_slot) == g["final_expert_of_slot"]


class MoveToFrontLRU:
    """Second formulation: a recency list of slots, oldest first.  Slots touched
    in one step move to the back in slot-index order (they share a timestamp)."""

    def __init__(self, n):
        self.order = list(range(n))
        self.expert = [-1] * n

    def step(self, ids):
        k = len(ids)
        hit, slot, ev = [0] * k, [-1] * k, [-1] * k
        touched = set()
        for j, e in enumerate(ids):
            if e in self.expert:
                s = self.expert.index(e)
                hit[j], slot[j] = 1, s
                touched.add(s)
        for j, e in enumerate(ids):
            if hit[j]:
                continue
            s = next(s for s in self.order if s not in touched)
            ev[j] = self.expert[s]
            self.expert[s] = e
            slot[j] = s
            touched.add(s)
        self.order = [s for s in self.order if s not in touched] + sorted(touched)
        return hit, slot, ev


def test_lru_agrees_with_move_to_front_formulation():
    rng = np.random.default_rng(10)
    for trial in range(100):
        E = int(rng.integers(3, 20))
        k = int(rng.integers(1, min(E, 6) + 1))
        n = int(rng.integers(k, E + 1))
        a, b = oracle.LRU(n), MoveToFrontLRU(n)
        for t in range(100):
            ids = rng.choice(E, size=k, replace=False).astype(np.int32)
            h1, s1, e1 = a.step(ids, t)
            h2, s2, e2 = b.step(list(ids))
            assert list(h1) == h2 and list(s1) == s2 and list(e1) == e2
        assert list(a.expert_of_slot) == b.expert


def test_lru_rejects_fewer_slots_than_k():
    with pytest.raises(ValueError):
        oracle.LRU(1).step([0, 1], 0)


# ----------------------------------------------------------------- LFU slot cache

def test_lfu_hand_worked_traces():
    with open(os.path.join(GOLDEN, "lfu_hand_traces.json")) as fh:
        g = json.load(fh)
    for tr in g["traces"]:
        lfu = oracle.LFU(tr["n_slots"], tr["n_experts"])
        hits = misses = 0
        for st in tr["steps"]:
            hit, slot, ev = lfu.step(st["ids"], st["t"])
            assert list(hit) == st["hit"], st
            assert list(slot) == st["slot"], st
            assert list(ev) == st["evicted"], st
            hits += int(hit.sum())
            misses += int(len(hit) - hit.sum())
        assert hits == tr["total_hits"] and misses == tr["total_misses"]
        assert list(lfu.expert_of_slot) == tr["final_expert_of_slot"]
        assert list(lfu.use_count) == tr["final_use_count"]


def test_lfu_reduces_to_lru_when_no_expert_repeats():
    """If no expert is picked twice, every cached expert has count 1 and the
    eviction order falls back to (last_use, slot): exactly LRU."""
    rng = np.random.default_rng(11)
    for trial in range(50):
        k = int(rng.integers(1, 5))
        n = int(rng.integers(k, 12))
        steps = 30
        E = steps * k
        seq = rng.permutation(E).astype(np.int32).reshape(steps, k)
        a, b = oracle.LFU(n, E), oracle.LRU(n)
        for t in range(steps):
            h1, s1, e1 = a.step(seq[t], t)
            h2, s2, e2 = b.step(seq[t], t)
            assert list(h1) == list(h2) and list(s1) == list(s2) and list(e1) == list(e2)


def test_lfu_keeps_a_hot_expert_through_a_scan():
    """A hot expert picked often survives a scan of one-off experts under LFU,
    and is evicted by it under LRU."""
    n, E = 4, 64
    lfu, lru = oracle.LFU(n, E), oracle.LRU(n)
    t = 0
    for _ in range(5):
        for pol in (lfu, lru):
            pol.step([7], t)
        t += 1
    for e in range(20, 30):
        for pol in (lfu, lru):
            pol.step([e], t)
        t += 1
    assert 7 in list(lfu.expert_of_slot)
    assert 7 not in list(lru.expert_of_slot)


def test_thread_count_does_not_change_results():
    # the rows of each matrix-vector product may run on several threads; every
    # row is still summed in index order by one thread, so results are bitwise
    # the same at any thread count
    sh = Shape(d=256, f=128, f_shared=192, n_experts=8, top_k=2)
    lay = oracle.Layer(gen_layer(sh, seed=77, layer=0), sh.top_k)
    x = oracle.rmsnorm_bf16(oracle.as_bits(gen_hidden(1, sh.d, seed=77)[0]), 1e-6)
    try:
        oracle.set_threads(1)
        ref = lay.forward(x, None)
        assert oracle.set_threads(4) in (1, 4)
        got = lay.forward(x, None)
    finally:
        oracle.set_threads(1)
    assert list(ref[0]) == list(got[0])
    assert np.array_equal(ref[3], got[3])
