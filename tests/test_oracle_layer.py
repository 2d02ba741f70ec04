"""Pins of the oracle's router, permutation and expert FFN / layer composition.

What pins each routine (none of these re-types the oracle's own code):
  * route: logits built to be exact, scores against sqrt(ln(1 + e^l)) evaluated in 40-digit
    arithmetic, top-k by full sort vs repeated arg-max, sum of weights = route
    scale, margin recomputed from the scores;
  * permute: an independent numpy stable sort of (expert, token) pairs, bijection, offsets;
  * expert FFN and layer: the hand-worked example in tests/golden/hand_worked_layer.json, exact
    symmetries (negated up projection, doubled down scale), reductions (E = 1, zero routed weights,
    no shared expert), dense per-token evaluation vs the permuted evaluation bit for bit.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_layer.json")


def _bf16_bits(v):
    a = np.asarray(v, dtype=np.float32).view(np.uint32)
    return ((a + 0x7FFF + ((a >> 16) & 1)) >> 16).astype(np.uint16)


def _pack_e2m1(values):
    """values on the E2M1 grid (scale 1) -> codes with element 2i in the low nibble of byte i."""
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    codes = []
    for v in values:
        c = grid.index(abs(v))
        codes.append(c | (8 if v < 0 else 0))
    codes = np.array(codes, dtype=np.uint8)
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def _hand_worked_inputs():
    g = json.load(open(GOLDEN))
    d, f = g["d"], g["f"]
    x = np.zeros((1, d), dtype=np.float32)
    for k, v in g["x_nonzero"].items():
        x[0, int(k)] = v
    xb = _bf16_bits(x)
    rw = np.zeros((2, d), dtype=np.float32)
    rw[1, 0] = g["router_w1_col0"]
    bias = np.zeros((2,), dtype=np.float32)
    # one expert's gate-up rows [2f, d] and down rows [d, f]
    w13 = np.zeros((2 * f, d))
    for o, (a, b) in g["gate_rows"].items():
        w13[int(o), :2] = [a, b]
    for o, (a, b) in g["up_rows"].items():
        w13[f + int(o), :2] = [a, b]
    w2 = np.zeros((d, f))
    for o, cols in g["down_rows"].items():
        for j, v in cols.items():
            w2[int(o), int(j)] = v
    s2 = np.full((d, f // 32), 127, dtype=np.uint8)
    for o, b in g["down_row_scale_bytes"].items():
        s2[int(o), :] = b
    expert = synth.ExpertWeights(
        np.stack([_pack_e2m1(r) for r in w13])[None], np.full((1, 2 * f, d // 32), 127, np.uint8),
        np.stack([_pack_e2m1(r) for r in w2])[None], s2[None])
    zero = synth.ExpertWeights(np.zeros_like(expert.w13), expert.s13.copy(), np.zeros_like(expert.w2), expert.s2.copy())
    routed = synth.ExpertWeights(*(np.concatenate([getattr(zero, n), getattr(expert, n)]) for n in ("w13", "s13", "w2", "s2")))
    return g, xb, rw, bias, routed, expert


def test_hand_worked_layer():
    g, xb, rw, bias, routed, shared = _hand_worked_inputs()
    e = g["expected"]
    q, s = oracle.quantize_x(xb)
    assert s[0, 0] == e["x_scale_byte"] and list(q[0, :2]) == e["x_codes_01"]
    ids, wts, margin, logits, scores = oracle.route(xb, rw, bias, k=1, want_logits=True)
    assert list(ids[0]) == e["ids"] and list(wts[0]) == e["weights"]
    assert np.allclose(scores[0], e["scores"], rtol=0, atol=1e-15)
    assert abs(margin[0] - (e["scores"][1] - e["scores"][0])) < 1e-15
    y1, hq, hs, hpre = oracle.expert_row(q[0], s[0], routed.w13[1], routed.s13[1], routed.w2[1], routed.s2[1])
    assert np.allclose(hpre[:4], e["h_pre"], rtol=1e-15, atol=0) and np.all(hpre[4:] == 0)
    assert hs[0] == e["h_scale_byte"]
    assert list(oracle.mxfp8_dequantize(hq, hs)[:4]) == e["h_dequant"]
    assert list(y1[:4]) == e["y_expert"] and np.all(y1[4:] == 0)
    for mode in (0, 1):
        y = oracle.layer(xb, ids, wts, routed, shared, mode=mode)
        assert list(y[0, :4]) == e["y"] and np.all(y[0, 4:] == 0)


def test_scores_against_direct_softplus():
    # x = e_0 in bf16 and router row e = [l_e, 0, ...] make the logits exactly l_e
    d, E = 64, 9
    ls = np.array([-20, -3, -0.5, 0, 0.25, 1, 2.5, 7, 30], dtype=np.float32)
    x = np.zeros((1, d), dtype=np.float32)
    x[0, 0] = 1.0
    rw = np.zeros((E, d), dtype=np.float32)
    rw[:, 0] = ls
    ids, wts, margin, logits, scores = oracle.route(_bf16_bits(x), rw, np.zeros(E, np.float32), k=3, want_logits=True)
    assert np.array_equal(logits[0], ls.astype(np.float64))
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    want = np.array([float(mpmath.sqrt(mpmath.log(1 + mpmath.exp(mpmath.mpf(float(l)))))) for l in ls])
    assert np.allclose(scores[0], want, rtol=4e-16, atol=0)
    assert list(ids[0]) == [6, 7, 8]
    assert np.allclose(wts[0], 1.5 * want[6:] / want[6:].sum(), rtol=1e-15)


def test_bias_changes_selection_not_weights():
    d, E = 32, 4
    x = np.zeros((1, d), dtype=np.float32)
    x[0, 0] = 1.0
    rw = np.zeros((E, d), dtype=np.float32)
    rw[:, 0] = [2.0, 1.0, 0.0, -1.0]
    bias = np.array([0.0, 0.0, 0.0, 5.0], dtype=np.float32)   # pushes expert 3 into the top-2
    ids, wts, margin, _, s = oracle.route(_bf16_bits(x), rw, bias, k=2, want_logits=True)
    assert list(ids[0]) == [0, 3]
    assert np.allclose(wts[0], 1.5 * s[0, [0, 3]] / (s[0, 0] + s[0, 3]), rtol=1e-15)
    # margin: sel = s + bias; 2nd largest is expert 0 (s0), 3rd is expert 1
    assert abs(margin[0] - (s[0, 0] - s[0, 1])) < 1e-15


def test_topk_sort_vs_selection_and_weight_sum():
    rng = np.random.default_rng(11)
    T, d, E, k = 64, 128, 32, 6
    x = _bf16_bits(rng.standard_normal((T, d)))
    rw = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    ids0, w0, m0, _, s = oracle.route(x, rw, bias, k, method=0, want_logits=True)
    ids1, w1, m1 = oracle.route(x, rw, bias, k, method=1)
    assert np.array_equal(ids0, ids1) and np.array_equal(w0, w1)
    assert np.all(np.abs(w0.sum(axis=1) - 1.5) < 1e-12)
    assert np.all(np.diff(ids0, axis=1) > 0)
    sel = s + bias.astype(np.float64)
    order = np.sort(sel, axis=1)[:, ::-1]
    assert np.allclose(m0, order[:, k - 1] - order[:, k], rtol=0, atol=1e-15)
    want_ids = np.sort(np.argsort(-sel, axis=1, kind="stable")[:, :k], axis=1)
    assert np.array_equal(ids0, want_ids)


def test_hash_route():
    tab = synth.gen_hash_table(0, 1000, 256, 6)
    assert all(len(set(r)) == 6 for r in tab) and tab.min() >= 0 and tab.max() < 256
    tok = synth.gen_token_ids(0, 50, 1000)
    ids, wts = oracle.hash_route(tok, tab, 6)
    assert np.array_equal(ids, np.sort(tab[tok], axis=1))
    assert np.all(wts == 0.25)


def test_permutation_against_stable_sort():
    rng = np.random.default_rng(5)
    T, E, k = 300, 17, 4
    ids = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    counts, offsets, perm, inv = oracle.permute(ids, E)
    pairs_e = ids.reshape(-1)
    pairs_t = np.repeat(np.arange(T), k)
    order = np.lexsort((pairs_t, pairs_e))           # expert-major, ascending token
    assert np.array_equal(perm, pairs_t[order])
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    assert np.array_equal(inv.reshape(-1), pos)
    assert counts.sum() == T * k and np.array_equal(counts, np.bincount(pairs_e, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(inv.reshape(-1)), np.arange(T * k))   # bijection
    for t in range(T):
        for j in range(k):
            r = inv[t, j]
            assert perm[r] == t and offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]


def _tiny_layer():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.gen_layer(wl, seed=0)
    ids, wts, _ = oracle.route_inputs(inp)
    return wl, inp, ids, wts


def test_dense_equals_permuted_bitwise():
    wl, inp, ids, wts = _tiny_layer()
    y0 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, mode=0)
    y1 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, mode=1)
    assert np.array_equal(y0, y1)
    sel = np.array([3, 0, 15, 7])
    y2 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, tokens=sel, mode=1)
    assert np.array_equal(y2, y0[sel])


def test_layer_h_outputs_are_the_rows_of_each_token_slot():
    """layer(want_h=True) returns, for every (token, slot), the h of that token through that slot's expert
    (slot k: the shared expert), the same in both evaluation orders, and y unchanged."""
    wl, inp, ids, wts = _tiny_layer()
    y = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared)
    sel = np.array([5, 0, 11])
    q, s = oracle.quantize_x(inp.x)
    for mode in (0, 1):
        y1, hq, hs, hp = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, tokens=sel, mode=mode, want_h=True)
        assert np.array_equal(y1, y[sel])
        assert hq.shape == (3, wl.k + 1, wl.f) and hs.shape == (3, wl.k + 1, wl.f // 32)
        for i, t in enumerate(sel):
            for j in range(wl.k + 1):
                src = inp.shared if j == wl.k else inp.experts
                e = 0 if j == wl.k else ids[t, j]
                _, hq_o, hs_o, hp_o = oracle.expert_row(q[t], s[t], src.w13[e], src.s13[e], src.w2[e], src.s2[e])
                assert np.array_equal(hq[i, j], hq_o) and np.array_equal(hs[i, j], hs_o)
                assert np.array_equal(hp[i, j], hp_o)


def test_reductions():
    wl, inp, ids, wts = _tiny_layer()
    # no shared expert: y = routed part only; routed weights zero: y = shared only
    y = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared)
    y_routed = oracle.layer(inp.x, ids, wts, inp.experts, None)
    y_shared = oracle.layer(inp.x, ids, np.zeros_like(wts), inp.experts, inp.shared)
    assert np.allclose(y, y_routed + y_shared, rtol=1e-13, atol=1e-13)
    # E = 1, k = 1: the weight is route_scale exactly, y = 1.5 FFN(x) + shared(x)
    one = synth.ExpertWeights(inp.experts.w13[:1], inp.experts.s13[:1], inp.experts.w2[:1], inp.experts.s2[:1])
    ids1, w1, _ = oracle.route(inp.x, inp.router_w[:1], inp.router_bias[:1], k=1)
    assert np.all(ids1 == 0) and np.allclose(w1, 1.5, rtol=2e-16, atol=0)
    y1 = oracle.layer(inp.x, ids1, w1, one, None)
    q, s = oracle.quantize_x(inp.x)
    yf, _, _ = oracle.expert_ffn(q, s, one)
    assert np.allclose(y1, 1.5 * yf, rtol=1e-15, atol=1e-300)


def test_exact_symmetries_of_the_expert():
    wl, inp, ids, wts = _tiny_layer()
    q, s = oracle.quantize_x(inp.x)
    e0 = synth.ExpertWeights(inp.experts.w13[:1], inp.experts.s13[:1], inp.experts.w2[:1], inp.experts.s2[:1])
    y, hq, hs = oracle.expert_ffn(q, s, e0)
    # doubling every down scale doubles y exactly
    e_d = synth.ExpertWeights(e0.w13, e0.s13, e0.w2, (e0.s2 + 1).astype(np.uint8))
    y_d, _, _ = oracle.expert_ffn(q, s, e_d)
    assert np.array_equal(y_d, 2 * y)
    # negating every up weight (flip code sign bits of rows f..2f-1) negates h and y exactly
    f = wl.f
    w13n = e0.w13.copy()
    w13n[:, f:] ^= 0x88
    y_n, hq_n, _ = oracle.expert_ffn(q, s, synth.ExpertWeights(w13n, e0.s13, e0.w2, e0.s2))
    assert np.array_equal(y_n, -y)
    # gate rows zero -> silu(0) = 0 -> h = 0 -> y = 0
    w13z = e0.w13.copy()
    w13z[:, :f] = 0
    y_z, hq_z, hs_z = oracle.expert_ffn(q, s, synth.ExpertWeights(w13z, e0.s13, e0.w2, e0.s2))
    assert np.all(y_z == 0) and np.all(hs_z == 0)


def test_clamp_engages_on_large_inputs():
    # x scaled by 30 makes |gate| and |up| exceed the limit 10; the clamp bounds |h| by
    # max silu(z) over z <= 10 times 10 = silu(10) * 10
    wl = synth.WORKLOADS["tiny"]
    inp = synth.gen_layer(wl, seed=1)
    x30 = synth.gen_x(1, wl.T, wl.d, scale=30.0)
    q, s = oracle.quantize_x(x30)
    e0 = synth.ExpertWeights(inp.experts.w13[:1], inp.experts.s13[:1], inp.experts.w2[:1], inp.experts.s2[:1])
    big = 0
    for t in range(wl.T):
        _, _, _, hpre = oracle.expert_row(q[t], s[t], e0.w13[0], e0.s13[0], e0.w2[0], e0.s2[0])
        assert np.all(np.abs(hpre) <= 10.0 / (1 + math.exp(-10.0)) * 10.0 + 1e-12)
        big += int(np.sum(np.abs(hpre) > 50))
    assert big > 0  # the clamp region is actually exercised
