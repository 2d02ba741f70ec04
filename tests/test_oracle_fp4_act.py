"""Pins of the oracle's MXFP4-activation variant (x and h quantised to MXFP4 instead of MXFP8).

What pins it (none of these re-types the oracle's own code):
  * the hand-worked example in tests/golden/hand_worked_layer_mxfp4.json (same inputs as the MXFP8
    example, quantised by hand);
  * activation quantisation against a brute-force nearest-grid-value search with the scale rule
    computed from math.frexp;
  * one-hot activations in even and odd positions: h before quantisation equals the closed form
    silu(min(W1[o, i] v, L)) * clamp(W3[o, i] v) from the dequantised weights (fixes the nibble order
    and the scale of the activation codes);
  * the down projection against a numpy matmul of the dequantised h codes and weights, and the h
    codes against the (separately pinned) MXFP4 quantiser applied to h before quantisation;
  * dense per-token evaluation vs the permuted evaluation, bit for bit.
"""
import json
import math
import os

import numpy as np

import oracle
import synth
from test_oracle_layer import _hand_worked_inputs

GOLDEN4 = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_layer_mxfp4.json")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _brute_e2m1(v: float) -> int:
    """Nearest E2M1 code by search over the grid, ties to the even mantissa (the even code), saturating."""
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(GRID[c] - a), c & 1))
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def _brute_mxfp4_block(vals):
    amax = max(abs(v) for v in vals)
    if amax == 0:
        se = -127
    else:
        m, e = math.frexp(amax)  # amax = m 2^e, 0.5 <= m < 1
        se = max(-127, min(127, (e - 1) - 2))
    codes = [_brute_e2m1(math.ldexp(v, -se)) for v in vals]
    return se + 127, codes


def test_hand_worked_layer_mxfp4():
    g, xb, rw, bias, routed, shared = _hand_worked_inputs()
    e = json.load(open(GOLDEN4))["expected"]
    q, s = oracle.quantize_x(xb, act="mxfp4")
    assert q.shape == (1, 16) and s[0, 0] == e["x_scale_byte"] and q[0, 0] == e["x_code_byte0"]
    assert np.all(q[0, 1:] == 0)
    ids, wts, _ = oracle.route(xb, rw, bias, k=1)
    y1, hq, hs, hpre = oracle.expert_row(q[0], s[0], routed.w13[1], routed.s13[1], routed.w2[1], routed.s2[1],
                                         act="mxfp4")
    assert hq.shape == (16,)
    assert np.allclose(hpre[:4], e["h_pre"], rtol=1e-15, atol=0) and np.all(hpre[4:] == 0)
    assert hs[0] == e["h_scale_byte"]
    assert list(oracle.mxfp4_dequantize(hq, hs)[:4]) == e["h_dequant"]
    assert list(y1[:4]) == e["y_expert"] and np.all(y1[4:] == 0)
    for mode in (0, 1):
        y = oracle.layer(xb, ids, wts, routed, shared, mode=mode, act="mxfp4")
        assert list(y[0, :4]) == e["y"] and np.all(y[0, 4:] == 0)


def test_activation_quantisation_matches_brute_force():
    x = synth.gen_x(3, 4, 256)
    x[1, :32] = 0                                   # an all-zero block
    x[2, 32:64] = np.uint16(0x8000)                 # negative zeros
    xs = synth.gen_x(4, 1, 256, scale=1e-30)        # tiny values (scale clamp region of E8M0 not reached)
    x = np.concatenate([x, xs])
    q, s = oracle.quantize_x(x, act="mxfp4")
    xf = _bf16_to_f64(x)
    for t in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            sb, codes = _brute_mxfp4_block(list(xf[t, 32 * b:32 * b + 32]))
            assert s[t, b] == sb
            got = [(q[t, 16 * b + i // 2] >> (4 * (i & 1))) & 15 for i in range(32)]
            assert got == codes, (t, b)


def _tiny():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.gen_layer(wl, seed=2)
    return wl, inp


def _deq_rows(codes, scales):
    return oracle.mxfp4_dequantize(codes, scales)


def test_one_hot_activations_fix_the_nibble_order():
    wl, inp = _tiny()
    d, f = wl.d, wl.f
    e0 = synth.ExpertWeights(inp.experts.w13[:1], inp.experts.s13[:1], inp.experts.w2[:1], inp.experts.s2[:1])
    w13 = _deq_rows(e0.w13[0], e0.s13[0])            # [2f, d]
    for i, v in ((0, 1.5), (1, -3.0), (36, 0.75), (255, 4.0)):
        x = np.zeros((1, d), dtype=np.float64)
        x[0, i] = v
        xb = oracle.bf16_encode(x)
        q, s = oracle.quantize_x(xb, act="mxfp4")
        assert oracle.mxfp4_dequantize(q, s)[0, i] == v   # a lone value is exact in MXFP4
        _, _, _, hpre = oracle.expert_row(q[0], s[0], e0.w13[0], e0.s13[0], e0.w2[0], e0.s2[0], act="mxfp4")
        g = w13[:f, i] * v
        u = w13[f:, i] * v
        gc = np.minimum(g, 10.0)
        want = gc / (1.0 + np.exp(-gc)) * np.clip(u, -10.0, 10.0)
        assert np.allclose(hpre, want, rtol=1e-14, atol=1e-300), i


def test_down_projection_and_h_codes():
    wl, inp = _tiny()
    q, s = oracle.quantize_x(inp.x, act="mxfp4")
    offsets = np.array([0, 5, 9, 16], dtype=np.int32)
    ex = synth.ExpertWeights(*(getattr(inp.experts, n)[:3] for n in ("w13", "s13", "w2", "s2")))
    row_w = np.linspace(0.5, 2.0, 16)
    y, hq, hs, hpre = oracle.expert_ffn(q, s, ex, offsets=offsets, row_w=row_w, act="mxfp4", want_hpre=True)
    assert hq.shape == (16, wl.f // 2)
    hq2, hs2 = oracle.mxfp4_quantize(hpre)
    assert np.array_equal(hq, hq2) and np.array_equal(hs, hs2)
    hd = oracle.mxfp4_dequantize(hq, hs)
    for g in range(3):
        w2 = _deq_rows(ex.w2[g], ex.s2[g])           # [d, f]
        rows = slice(offsets[g], offsets[g + 1])
        want = (hd[rows] @ w2.T) * row_w[rows, None]
        assert np.allclose(y[rows], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_down_from_h_equals_the_ffn_down_projection():
    """oracle.down_from_h on the oracle's own h reproduces expert_ffn's y (both formats)."""
    wl, inp = _tiny()
    ex = synth.ExpertWeights(*(getattr(inp.experts, n)[:1] for n in ("w13", "s13", "w2", "s2")))
    for act in ("mxfp8", "mxfp4"):
        q, s = oracle.quantize_x(inp.x, act=act)
        y, hq, hs = oracle.expert_ffn(q, s, ex, act=act)
        y2 = oracle.down_from_h(hq, hs, ex.w2[0], ex.s2[0], act=act)
        assert np.allclose(y2, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_dense_equals_permuted_bitwise_mxfp4():
    wl, inp = _tiny()
    ids, wts, _ = oracle.route_inputs(inp)
    y0 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, mode=0, act="mxfp4")
    y1 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, mode=1, act="mxfp4")
    assert np.array_equal(y0, y1)
    # the variant really quantises differently from the MXFP8 layer, and stays close to it
    y8 = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, mode=1)
    rel = np.abs(y1 - y8).sum() / np.abs(y8).sum()
    assert 1e-3 < rel < 0.5
