"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Integer and byte results are compared bit for bit: expert ids, counts, offsets, the permutation and
its inverse, the MXFP8 activation codes and scale bytes.  The layer output is checked in two steps:
the fp32 sums the combine rounds (read back with moe_testing_read_y32) against the layer's contract
exactly as written (max |dy| <= 2e-2 rms, mean relative error <= 5e-3), and the bf16 output against
those sums rounded to nearest even, bit for bit.  The MXFP8 h codes the down projection consumed are
compared with the oracle's, code by code, except at rounding midpoints the two precisions may
straddle.  Every token row is compared for the small workloads and for verify8, verify512 and
hash512; at prefill8192 at least 512 tokens, chosen so that every 128-row tile of every expert group
(the shared expert's included) holds a compared row, plus the bit-exact rounding check on all rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from gpu_support import (BF16_HALF_ULP_REL, TOL_MAX_RMS, TOL_WEIGHT_REL, WORKLOADS, assert_close, assert_strict, bf16_to_f64, case, check_h8, device,
                         forward_strict, gpu_h_by_slot, x_to_device)

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "medium", "wide"]
FULL = ["verify8", "verify512", "hash512", "prefill8192"]


def _routing_on_gpu(layer, x):
    ids, w = layer.route(x)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", SMALL + FULL)
def test_route_parity(name):
    wl, inp, ids_ref, wts_ref, layer = case(name)
    x = x_to_device(inp.x)
    ids, w = _routing_on_gpu(layer, x)
    layer.check()
    assert np.array_equal(ids, ids_ref)
    assert np.max(np.abs(w - wts_ref) / np.abs(wts_ref)) <= TOL_WEIGHT_REL
    assert np.allclose(w.sum(axis=1), wl.route_scale, rtol=1e-5)


@pytest.mark.parametrize("name,T", [("wide", 16), ("wide", 32), ("verify512", 32), ("verify512", 33)])
def test_route_parity_small_batch_boundary(name, T):
    """Batches of up to 32 rows take the small-batch router (fp32 logits over the whole GPU, top-k in its
    last CTA), larger ones the tensor-core cluster router: both sides of the boundary, 256 and 384 experts."""
    wl, inp, ids_ref, wts_ref, layer = case(name, T=T)
    ids, w = _routing_on_gpu(layer, x_to_device(inp.x))
    layer.check()
    assert np.array_equal(ids, ids_ref)
    assert np.max(np.abs(w - wts_ref) / np.abs(wts_ref)) <= TOL_WEIGHT_REL
    # twice in a row: the kernel's CTA count is back at zero
    ids2, w2 = _routing_on_gpu(layer, x_to_device(inp.x))
    assert np.array_equal(ids2, ids) and np.array_equal(w2, w)


@pytest.mark.parametrize("name", SMALL + FULL)
def test_permute_parity(name):
    wl, inp, ids_ref, wts_ref, layer = case(name)
    x = x_to_device(inp.x)
    out = layer.permute(x, torch.from_numpy(ids_ref).to(device()))
    torch.cuda.synchronize()
    layer.check()
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["perm_tok"].cpu().numpy(), perm)
    assert np.array_equal(out["inv_pos"].cpu().numpy(), inv)
    q, s = oracle.quantize_x(inp.x)
    assert np.array_equal(out["a_q"].cpu().numpy(), q[perm])
    assert np.array_equal(out["a_s"].cpu().numpy(), s[perm])


def _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, tokens=None, what=""):
    """Forward the whole batch; for the listed tokens (None: all) check the fp32 sums strictly against the
    oracle and the h codes of each token's k + 1 rows; the bf16 output is checked on every row."""
    x = x_to_device(inp.x)
    y, y32 = forward_strict(layer, x)
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    toks = np.arange(wl.T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
    y_ref, hq_ref, hs_ref, hpre = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit,
                                               tokens=None if tokens is None else toks, want_h=True)
    assert_strict(y32.cpu().numpy().astype(np.float64)[toks], y_ref, f"{what} fp32 sums")
    hq, hs = (t.cpu().numpy() for t in layer.last_h())
    _, _, _, inv = oracle.permute(ids_ref, wl.E)
    hq_d, hs_d = gpu_h_by_slot(hq, hs, inv, toks, wl.T * wl.k)
    f = wl.f
    check_h8(hq_d.reshape(-1, f), hs_d.reshape(-1, f // 32), hq_ref.reshape(-1, f), hs_ref.reshape(-1, f // 32),
             hpre.reshape(-1, f), f"{what} h")
    return y


@pytest.mark.parametrize("name", SMALL)
def test_forward_elementwise(name):
    wl, inp, ids_ref, wts_ref, layer = case(name)
    _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=name)


def tile_covering_tokens(ids, E, T, tile_rows=128, n_min=512, seed=1):
    """Tokens such that every row tile of every expert group holds one of them: for each routed group,
    one random row of each run of tile_rows rows in its permuted order (so every hot expert's tiles and
    every cold expert), one token of each tile_rows-token run of the shared group, then random tokens up
    to n_min; plus the first and the last token."""
    rng = np.random.default_rng(seed)
    counts, offsets, perm, _ = oracle.permute(ids, E)
    picks = [0, T - 1]
    for g in range(E):
        for r0 in range(offsets[g], offsets[g + 1], tile_rows):
            r1 = min(r0 + tile_rows, offsets[g + 1])
            picks.append(int(perm[rng.integers(r0, r1)]))
    for t0 in range(0, T, tile_rows):
        picks.append(int(rng.integers(t0, min(t0 + tile_rows, T))))
    toks = np.unique(picks)
    if toks.size < n_min:
        rest = np.setdiff1d(np.arange(T), toks)
        toks = np.unique(np.concatenate([toks, rng.choice(rest, n_min - toks.size, replace=False)]))
    return toks.astype(np.int32)


@pytest.mark.parametrize("name", ["verify8", "verify512", "hash512"])
def test_forward_full_size_every_row(name):
    """The decode-shape workloads in the configuration the benchmark times, every token row."""
    wl, inp, ids_ref, wts_ref, layer = case(name)
    y = _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=name)
    y2 = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    assert torch.equal(y, y2)  # repeatable bit for bit


def test_forward_prefill_tile_covering_rows():
    """prefill8192 (26 hot experts with thousands of rows, cold experts with one or a few, 8192 shared
    rows): at least 512 tokens covering every 128-row tile of every group, compared strictly; the bf16
    rounding is checked on all 8192 rows."""
    wl, inp, ids_ref, wts_ref, layer = case("prefill8192")
    toks = tile_covering_tokens(ids_ref, wl.E, wl.T)
    assert toks.size >= 512
    y = _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, tokens=toks, what="prefill8192")
    y2 = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("name", SMALL)
def test_expert_ffn_stage(name):
    """moe_expert_ffn on the oracle's own permuted MXFP8 rows: grouped FFN of the routed experts, and
    the shared expert over the token-order rows."""
    wl, inp, ids_ref, wts_ref, layer = case(name)
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    q, s = oracle.quantize_x(inp.x)
    a_q, a_s = q[perm], s[perm]
    row_w = np.empty(perm.shape[0])
    row_w[inv.reshape(-1)] = wts_ref.reshape(-1)
    dev = device()
    y = layer.expert_ffn(torch.from_numpy(a_q).to(dev), torch.from_numpy(a_s).to(dev),
                         torch.from_numpy(offsets).to(dev), torch.from_numpy(row_w.astype(np.float32)).to(dev))
    torch.cuda.synchronize()
    layer.check()
    y_ref, hq_ref, hs_ref, hpre = oracle.expert_ffn(a_q, a_s, inp.experts, offsets=offsets, row_w=row_w,
                                                    want_hpre=True)
    assert_close(bf16_to_f64(y), y_ref, f"{name} routed FFN")
    hq, hs = (t.cpu().numpy() for t in layer.last_h())
    check_h8(hq, hs, hq_ref, hs_ref, hpre, f"{name} routed FFN h")
    ys = layer.expert_ffn(torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev), shared=True)
    torch.cuda.synchronize()
    ys_ref, _, _ = oracle.expert_ffn(q, s, inp.shared)
    assert_close(bf16_to_f64(ys), ys_ref, f"{name} shared FFN")


def test_expert_ffn_wide_weight_scales():
    """Weight E8M0 bytes far from the generator's two values, through moe_expert_ffn: expert 0 with
    every scale 40 binades above the usual (gate and up then pass the clamp), expert 1 with every scale
    20 below (kept where no product leaves fp32's normal range), expert 2 with a quarter of its gate
    and up rows at byte 0x00 (2^-127) and the rest usual, experts 3..7 with every block's byte drawn
    from usual +-24.  Rows are compared one by one (each row within 2e-2 of its own rms plus its
    bf16 rounding), and the h codes against the oracle's."""
    wl = synth.Workload("wide_scales", 96, 512, 256, 8, 2)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=9)
    rng = np.random.default_rng(9)
    for name in ("s13", "s2"):
        sc = getattr(inp.experts, name).astype(np.int64)
        sc[0] += 40
        sc[1] -= 20
        sc[3:] += rng.integers(-24, 25, size=sc[3:].shape)
        if name == "s13":
            quarter = rng.permutation(2 * wl.f)[: wl.f // 2]
            sc[2, quarter] = 0
        assert sc.min() >= 0 and sc.max() <= 254
        setattr(inp.experts, name, sc.astype(np.uint8))
    layer = _layer_from(inp)
    try:
        counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
        assert np.all(counts[:3] > 0)
        q, s = oracle.quantize_x(inp.x)
        a_q, a_s = q[perm], s[perm]
        row_w = np.empty(perm.shape[0])
        row_w[inv.reshape(-1)] = wts_ref.reshape(-1)
        dev = device()
        y = layer.expert_ffn(torch.from_numpy(a_q).to(dev), torch.from_numpy(a_s).to(dev),
                             torch.from_numpy(offsets).to(dev), torch.from_numpy(row_w.astype(np.float32)).to(dev))
        torch.cuda.synchronize()
        layer.check()
        y_ref, hq_ref, hs_ref, hpre = oracle.expert_ffn(a_q, a_s, inp.experts, offsets=offsets, row_w=row_w,
                                                        want_hpre=True)
        yd = bf16_to_f64(y)
        assert np.all(np.isfinite(yd))
        rms_r = np.sqrt(np.mean(y_ref ** 2, axis=1, keepdims=True))
        err = np.abs(yd - y_ref)
        excess = err - (TOL_MAX_RMS * rms_r + BF16_HALF_ULP_REL * np.abs(y_ref))
        worst = int(np.argmax(excess.max(axis=1)))
        print(f"wide scales: worst row {worst} (expert {np.searchsorted(offsets, worst, 'right') - 1}): "
              f"max |dy| / row rms = {err[worst].max() / rms_r[worst, 0]:.3e}")
        assert np.all(excess <= 0), f"row {worst} exceeds its own tolerance by {excess.max():.3e}"
        # the construction reached the extremes: expert 0's rows are about 2^80 times expert 1's
        assert rms_r[: offsets[1]].min() > 1e9 * rms_r[offsets[1]:offsets[2]].max()
        hq, hs = (t.cpu().numpy() for t in layer.last_h())
        check_h8(hq, hs, hq_ref, hs_ref, hpre, "wide scales h")
    finally:
        layer.close()


@pytest.mark.parametrize("case", ["up60", "down60", "rows40"])
def test_forward_expert_rows_across_the_fp32_range(case):
    """The weighted expert rows travel from the down GEMM to the combine as fp16 with one power-of-two scale
    per 32 columns.  Drive them far outside fp16's own range and across a wide range inside one block, then
    compare the fp32 sums strictly with the oracle: every down scale byte (routed and shared) 60 binades up
    (rows near 2^60, far above fp16's 65504), 60 down (rows near 2^-60, far below its smallest normal), or
    each output row of W2 shifted by its own draw from -20..20 binades (columns inside one 32-column block
    of y then span up to 2^40)."""
    wl = WORKLOADS["tiny"].with_T(64)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=11)
    rng = np.random.default_rng(11)
    for ew in (inp.experts, inp.shared):
        sc = ew.s2.astype(np.int64)  # [n, d, f / 32]
        if case == "up60":
            sc += 60
        elif case == "down60":
            sc -= 60
        else:
            sc += rng.integers(-20, 21, size=sc.shape[:2])[:, :, None]
        assert sc.min() >= 1 and sc.max() <= 254
        ew.s2 = sc.astype(np.uint8)
    layer = _layer_from(inp)
    try:
        y = _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"rows {case}")
        assert torch.isfinite(y.float()).all()
        y_ref, _, _, _ = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit, want_h=True)
        mag = float(np.sqrt(np.mean(y_ref ** 2)))
        if case == "up60":
            assert mag > 2.0 ** 50
        elif case == "down60":
            assert mag < 2.0 ** -50
    finally:
        layer.close()


@pytest.mark.parametrize("T", [1024, 1025])
@pytest.mark.parametrize("routing", ["learned", "hash"])
def test_forward_at_the_dispatch_state_boundary(routing, T):
    """Up to 1024 rows the routing kernel's last CTA writes the dispatch state (chunk bases, counts, offsets,
    the tile list); above that the histogram and scan kernels do.  Both sides of the switch, for the cluster
    router and the hash router, every row against the oracle (d = 1024, f = 512, 16 experts top-4: about 256
    rows per expert, several 128-row tiles each)."""
    wl = synth.Workload(f"boundary_{routing}", T, 1024, 512, 16, 4, hash_vocab=4096 if routing == "hash" else 0)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=5)
    layer = _layer_from(inp)
    try:
        _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"{routing} T={T}")
        counts, _, _, _ = oracle.permute(ids_ref, wl.E)
        assert counts.min() > 128  # every expert group spans more than one 128-row tile
    finally:
        layer.close()


@pytest.mark.parametrize("name", ["tiny", "wide", "verify8", "verify512"])
def test_resident_router_matches_per_call_router(name):
    """moe_experts_set_router (weights split once on the handle) gives the per-call router's ids,
    weights and layer output bit for bit, through moe_route and moe_forward."""
    from block_scaled_fp4_sqrt_gb300 import moe_experts_set_router, moe_forward, moe_route
    wl, inp, ids_ref, wts_ref, layer = case(name)
    x = x_to_device(inp.x)
    y_call = layer.forward(x)
    ids_call, w_call = layer.route(x)
    moe_experts_set_router(layer.h, layer.router_w, layer.router_bias)
    try:
        ids = torch.empty_like(ids_call)
        w = torch.empty_like(w_call)
        moe_route(layer.h, x, None, None, ids, w)
        y = torch.empty_like(y_call)
        moe_forward(x, None, None, layer.h, layer.h_shared, y)
        torch.cuda.synchronize()
        layer.check()
        assert torch.equal(ids, ids_call) and torch.equal(w, w_call)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert torch.equal(y, y_call)
    finally:
        moe_experts_set_router(layer.h, None, None)


def test_resident_router_argument_checks():
    from block_scaled_fp4_sqrt_gb300 import MoEError, moe_experts_set_router, moe_forward
    wl, inp, ids_ref, wts_ref, layer = case("tiny")
    x = x_to_device(inp.x)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=device())
    with pytest.raises(MoEError):  # no resident router and no weights given
        moe_forward(x, None, None, layer.h, layer.h_shared, y)
    with pytest.raises(MoEError):  # weights without a bias
        moe_experts_set_router(layer.h, layer.router_w, None)
    mis = torch.empty(layer.router_w.numel() + 4, dtype=torch.float32, device=device())[1:1 + layer.router_w.numel()]
    with pytest.raises(MoEError):  # not 16-byte aligned
        moe_experts_set_router(layer.h, mis, layer.router_bias)
    moe_experts_set_router(layer.h, None, None)  # nothing resident: dropping is a no-op


@pytest.mark.parametrize("T", [1, 2, 31, 33, 100, 256])
def test_tiny_ragged_sizes(T):
    """Chunk / tile edges: one token, partial 32-token chunks, expert groups longer than a 32-row tile."""
    wl, inp, ids_ref, wts_ref, layer = case("tiny", T=T)
    _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"tiny T={T}")


@pytest.mark.parametrize("E,k,T", [(9, 2, 8), (9, 2, 40), (1, 1, 5), (1, 1, 37)])
def test_odd_and_single_expert_counts(E, k, T):
    """An odd expert count (the small-batch router's last CTA holds one expert) and a single expert with
    top-1, on both sides of the 32-row boundary: routing bit for bit, output within the tolerance."""
    wl = synth.Workload(f"e{E}k{k}", T, 256, 128, E, k)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=6)
    layer = _layer_from(inp)
    try:
        _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"E={E} k={k} T={T}")
    finally:
        layer.close()


def test_empty_batch():
    wl, inp, ids_ref, wts_ref, layer = case("tiny")
    x = torch.empty((0, wl.d), dtype=torch.bfloat16, device=device())
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    assert y.shape == (0, wl.d)


def _layer_from(inp, with_shared=True):
    from block_scaled_fp4_sqrt_gb300 import MoELayer
    return MoELayer.from_host(inp, device=device(), max_T=inp.wl.T, with_shared=with_shared)


def test_no_shared_expert_and_empty_experts():
    """No shared expert; and half of the routed experts never selected (their groups are empty)."""
    wl = WORKLOADS["tiny"].with_T(64)

    def starve(inp):
        inp.router_bias[:4] -= 50.0

    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=3, adjust=starve)
    assert ids_ref.min() >= 4
    layer = _layer_from(inp, with_shared=False)
    y, y32 = forward_strict(layer, x_to_device(inp.x))
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, None, wl.swiglu_limit)
    assert_strict(y32.cpu().numpy().astype(np.float64), y_ref, "no shared, empty experts")
    layer.close()


def test_swiglu_clamp_engaged():
    """x scaled by 30: gate and up pass the limit 10 for many features."""
    wl = WORKLOADS["tiny"].with_T(64)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=5, x_scale=30.0)
    layer = _layer_from(inp)
    _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what="clamped")
    layer.close()


def test_e4m3_activation_codes_exhaustive():
    """Every finite bf16 value through the MXFP8 quantiser (moe_permute), in blocks of mixed and of
    similar magnitudes, against the oracle's round-to-nearest-even encoder, byte for byte."""
    wl, inp, _, _, layer = case("tiny")
    bits = np.arange(65536, dtype=np.uint32)
    finite = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    rng = np.random.default_rng(0)
    d = wl.d
    n = (finite.size // d) * d
    mixed = rng.permutation(finite)[:n].reshape(-1, d)
    similar = np.sort(finite)[:n].reshape(-1, d)
    xb = np.concatenate([mixed, similar])
    T = xb.shape[0]
    ids = np.sort(np.stack([np.arange(T) % wl.E, (np.arange(T) + 3) % wl.E], axis=1), axis=1).astype(np.int32)
    from block_scaled_fp4_sqrt_gb300 import MoELayer
    big = MoELayer.from_host(inp, device=device(), max_T=T)
    out = big.permute(x_to_device(xb), torch.from_numpy(ids).to(device()))
    torch.cuda.synchronize()
    big.check()
    counts, offsets, perm, inv = oracle.permute(ids, wl.E)
    q, s = oracle.quantize_x(xb)
    assert np.array_equal(out["perm_tok"].cpu().numpy(), perm)
    assert np.array_equal(out["a_s"].cpu().numpy(), s[perm])
    assert np.array_equal(out["a_q"].cpu().numpy(), q[perm])
    big.close()


def test_hash_out_of_range_token_is_reported():
    from block_scaled_fp4_sqrt_gb300 import MoEError, MoELayer
    wl = synth.Workload("hashtiny", 16, 256, 128, 8, 2, hash_vocab=100)
    inp = synth.gen_layer(wl, seed=0)
    layer = MoELayer.from_host(inp, device=device(), max_T=16)
    tok = torch.from_numpy(inp.token_ids.copy()).to(device())
    y, y32 = forward_strict(layer, x_to_device(inp.x), token_ids=tok)  # in range: no error
    ids_ref, wts_ref = oracle.hash_route(inp.token_ids, inp.hash_table, wl.k, wl.route_scale)
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_strict(y32.cpu().numpy().astype(np.float64), y_ref, "hash tiny")
    tok[3] = 150
    layer.forward(x_to_device(inp.x), token_ids=tok)
    with pytest.raises(MoEError) as err:
        layer.check()
    assert err.value.status == 5
    layer.check()  # the status is cleared once read
    layer.close()


def test_bounded_wait_reports_timeout_and_context_survives():
    import block_scaled_fp4_sqrt_gb300 as m
    wl = WORKLOADS["tiny"].with_T(32)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=7)
    layer = _layer_from(inp)
    x = x_to_device(inp.x)
    m.moe_set_wait_budget(layer.h, 20_000_000)  # 20 ms
    m.moe_testing_stall_loads(layer.h, True)
    layer.forward(x)
    with pytest.raises(m.MoEError) as err:
        m.moe_check(layer.h)
    assert err.value.status == 6
    m.moe_testing_stall_loads(layer.h, False)
    m.moe_set_wait_budget(layer.h, 2_000_000_000)
    y, y32 = forward_strict(layer, x)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_strict(y32.cpu().numpy().astype(np.float64), y_ref, "after timeout")
    layer.close()


@pytest.mark.parametrize("name,T", [("medium", None), ("tiny", 256), ("tiny", 100)])
def test_cta_pair_and_one_sm_gemms_both_match_the_oracle(name, T):
    """Batches with 128-row tiles run their grouped GEMMs on the one-SM kernels by default, or on CTA pairs
    (M = 256 over two SMs) when the handle selects them.  Both meet the strict bound and give the same
    routing; the print shows how far apart their fp32 sums are (accumulation order)."""
    from block_scaled_fp4_sqrt_gb300 import moe_testing_set_pair_gemm
    wl, inp, ids_ref, wts_ref, layer = case(name, T=T)
    _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"{name} T={wl.T} one SM")
    y32_one = layer.last_y32()
    for h in (layer.h, layer.h_shared):
        moe_testing_set_pair_gemm(h, True)
    try:
        _strict_layer_parity(wl, inp, ids_ref, wts_ref, layer, what=f"{name} T={wl.T} CTA pair")
        y32_pair = layer.last_y32()
        torch.cuda.synchronize()
        d = (y32_pair - y32_one).abs().max().item() / y32_one.pow(2).mean().sqrt().item()
        print(f"{name} T={wl.T}: max |pair - one SM| / rms = {d:.3e}")
        assert d <= 2e-2
    finally:
        for h in (layer.h, layer.h_shared):
            moe_testing_set_pair_gemm(h, False)


def test_cta_pair_bounded_wait_reports_timeout_and_context_survives():
    """The CTA-pair GEMM's waits (the leader's stage and accumulator barriers, both CTAs' epilogues) run
    out when no loads are issued; the status reports it and the next forward is correct."""
    import block_scaled_fp4_sqrt_gb300 as m
    wl = WORKLOADS["tiny"].with_T(256)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=8)
    layer = _layer_from(inp)
    for h in (layer.h, layer.h_shared):
        m.moe_testing_set_pair_gemm(h, True)
    x = x_to_device(inp.x)
    m.moe_set_wait_budget(layer.h, 20_000_000)  # 20 ms
    m.moe_testing_stall_loads(layer.h, True)
    layer.forward(x)
    with pytest.raises(m.MoEError) as err:
        m.moe_check(layer.h)
    assert err.value.status == 6
    m.moe_testing_stall_loads(layer.h, False)
    m.moe_set_wait_budget(layer.h, 2_000_000_000)
    y, y32 = forward_strict(layer, x)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_strict(y32.cpu().numpy().astype(np.float64), y_ref, "CTA pair after timeout")
    layer.close()


def test_batch_above_workspace_is_rejected():
    from block_scaled_fp4_sqrt_gb300 import MoEError
    wl, inp, _, _, layer = case("tiny")
    x = torch.zeros((wl.T + 1, wl.d), dtype=torch.bfloat16, device=device())
    with pytest.raises(MoEError) as err:
        layer.forward(x)
    assert err.value.status == 3
