"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Integer and byte results are compared bit for bit: expert ids, counts, offsets, the permutation and
its inverse, the MXFP8 activation codes and scale bytes.  Floating-point results use the layer's
tolerance (max |dy| <= 2e-2 rms, mean relative error <= 5e-3) and, for the routing weights, a bound
derived from fp32 dot products.  Small workloads are compared element by element; the full-size
workloads (in the configuration the benchmark times) on sampled tokens plus all integer outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from gpu_support import (TOL_WEIGHT_REL, WORKLOADS, assert_close, bf16_to_f64, case, device, x_to_device)

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


@pytest.mark.parametrize("name", SMALL)
def test_forward_elementwise(name):
    wl, inp, ids_ref, wts_ref, layer = case(name)
    x = x_to_device(inp.x)
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, f"{name} forward")


def _sample_tokens(T, n=24, seed=1):
    rng = np.random.default_rng(seed)
    extra = rng.choice(T, size=min(n, T), replace=False)
    return np.unique(np.concatenate([[0, T - 1], extra])).astype(np.int32)


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(name):
    wl, inp, ids_ref, wts_ref, layer = case(name)
    x = x_to_device(inp.x)
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    toks = _sample_tokens(wl.T)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit, tokens=toks)
    assert_close(bf16_to_f64(y)[toks], y_ref, f"{name} forward (tokens {toks.tolist()})")
    # every output row is finite and the whole output repeats bit for bit on a second call
    y2 = layer.forward(x)
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
    y_ref, _, _ = oracle.expert_ffn(a_q, a_s, inp.experts, offsets=offsets, row_w=row_w)
    assert_close(bf16_to_f64(y), y_ref, f"{name} routed FFN")
    ys = layer.expert_ffn(torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev), shared=True)
    torch.cuda.synchronize()
    ys_ref, _, _ = oracle.expert_ffn(q, s, inp.shared)
    assert_close(bf16_to_f64(ys), ys_ref, f"{name} shared FFN")


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
    x = x_to_device(inp.x)
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, f"tiny T={T}")


@pytest.mark.parametrize("E,k,T", [(9, 2, 8), (9, 2, 40), (1, 1, 5), (1, 1, 37)])
def test_odd_and_single_expert_counts(E, k, T):
    """An odd expert count (the small-batch router's last CTA holds one expert) and a single expert with
    top-1, on both sides of the 32-row boundary: routing bit for bit, output within the tolerance."""
    wl = synth.Workload(f"e{E}k{k}", T, 256, 128, E, k)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=6)
    layer = _layer_from(inp)
    try:
        x = x_to_device(inp.x)
        y = layer.forward(x)
        torch.cuda.synchronize()
        layer.check()
        assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
        y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
        assert_close(bf16_to_f64(y), y_ref, f"E={E} k={k} T={T}")
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
    y = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    layer.check()
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, None, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, "no shared, empty experts")
    layer.close()


def test_swiglu_clamp_engaged():
    """x scaled by 30: gate and up pass the limit 10 for many features."""
    wl = WORKLOADS["tiny"].with_T(64)
    inp, ids_ref, wts_ref, _ = oracle.margin_filtered_layer(wl, seed=5, x_scale=30.0)
    layer = _layer_from(inp)
    y = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    layer.check()
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, "clamped")
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
    y = layer.forward(x_to_device(inp.x), token_ids=tok)
    torch.cuda.synchronize()
    layer.check()  # in range: no error
    ids_ref, wts_ref = oracle.hash_route(inp.token_ids, inp.hash_table, wl.k, wl.route_scale)
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, "hash tiny")
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
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    y_ref = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    assert_close(bf16_to_f64(y), y_ref, "after timeout")
    layer.close()


def test_batch_above_workspace_is_rejected():
    from block_scaled_fp4_sqrt_gb300 import MoEError
    wl, inp, _, _, layer = case("tiny")
    x = torch.zeros((wl.T + 1, wl.d), dtype=torch.bfloat16, device=device())
    with pytest.raises(MoEError) as err:
        layer.forward(x)
    assert err.value.status == 3
