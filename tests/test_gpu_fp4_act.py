"""The MXFP4-activation variant (x and h quantised to MXFP4, grouped GEMMs on tcgen05 kind::mxf4)
against the oracle run with the same activation format.

* Bytes bit for bit: moe_permute's MXFP4 activation codes and scales, for every finite bf16 value and
  for the workloads' x.
* h: the kernels quantise their fp32 h, the oracle its fp64 h, so an E2M1 code may differ only where
  the oracle's h lies within 2^-10 (in units of the block scale) of a rounding midpoint or of zero, or
  where the block maximum lies within 1e-4 (relative) of a power of two.  The kernels' h comes from
  fp32 sums of exact products; its relative error is orders of magnitude below those margins.  Every
  other code and scale byte must match the oracle's.
* Output: an E2M1 step is a third of a block's range, so one code flip moves a row by more than the
  layer's tolerance; the decision is the kernel's (taken in its precision).  The output is therefore
  compared, with the layer's tolerance, to the oracle's down projection and fixed-order combine
  evaluated on the kernels' own h codes.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from gpu_support import WORKLOADS, assert_close, bf16_to_f64, case, device, x_to_device

pytestmark = pytest.mark.gpu

ACT = "mxfp4"
MIDPOINTS = np.array([0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    return np.stack([p & 15, p >> 4], axis=-1).reshape(p.shape[:-1] + (p.shape[-1] * 2,))


def _fragile(hpre: np.ndarray, hs_ref: np.ndarray):
    """(code_fragile [n, f], scale_fragile [n, f/32]) from the oracle's h before quantisation."""
    n, f = hpre.shape
    blocks = hpre.reshape(n, f // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    scale_fragile = (amax > 0) & (np.abs(lg - np.round(lg)) <= 1.5e-4)
    unit = np.ldexp(1.0, hs_ref.astype(np.int64) - 127)[:, :, None]
    v = np.abs(blocks) / unit
    near = np.min(np.abs(v[..., None] - MIDPOINTS), axis=-1) <= 2.0 ** -10
    return near.reshape(n, f), scale_fragile


def check_h(hq_gpu, hs_gpu, hq_ref, hs_ref, hpre, what):
    """Codes and scales equal the oracle's except where the oracle's own h is fragile."""
    code_fragile, scale_fragile = _fragile(hpre, hs_ref)
    bad_scale = hs_gpu != hs_ref
    assert not np.any(bad_scale & ~scale_fragile), f"{what}: {int(np.sum(bad_scale & ~scale_fragile))} scale bytes differ"
    c_gpu, c_ref = _nibbles(hq_gpu), _nibbles(hq_ref)
    same_scale = np.repeat(~bad_scale, 32, axis=1)
    bad_code = (c_gpu != c_ref) & same_scale
    assert not np.any(bad_code & ~code_fragile), f"{what}: {int(np.sum(bad_code & ~code_fragile))} h codes differ"
    return int(bad_code.sum()) + 32 * int(bad_scale.sum())


def y_on_gpu_h(hq, hs, rows_expert, row_w, experts, shared, inv, T, R):
    """Token outputs from the device's h rows: routed rows through their experts (times row_w), then
    the shared rows; summed per token in slot order, then the shared row."""
    d = experts.w2.shape[1]
    yr = np.zeros((R, d))
    for e in np.unique(rows_expert):
        r = np.nonzero(rows_expert == e)[0]
        yr[r] = oracle.down_from_h(hq[r], hs[r], experts.w2[e], experts.s2[e], ACT) * row_w[r, None]
    ysh = oracle.down_from_h(hq[R:R + T], hs[R:R + T], shared.w2[0], shared.s2[0], ACT)
    y = yr[inv[:, 0]].copy()
    for j in range(1, inv.shape[1]):
        y = y + yr[inv[:, j]]
    return y + ysh


def test_mxf4_peak_is_measured():
    from block_scaled_fp4_sqrt_gb300 import moe_measure_mxf4_peak, moe_measure_mxf8f6f4_peak
    p4 = moe_measure_mxf4_peak(2048)
    p8 = moe_measure_mxf8f6f4_peak(2048)
    assert np.isfinite(p4) and p4 > 0 and np.isfinite(p8) and p8 > 0


def test_fp4_activation_codes_exhaustive():
    """Every finite bf16 value through the MXFP4 quantiser of moe_permute, in blocks of mixed and of
    similar magnitudes, against the oracle's E2M1 encoder and scale rule, byte for byte."""
    wl, inp, _, _, layer = case("tiny", act=ACT)
    bits = np.arange(65536, dtype=np.uint32)
    finite = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    rng = np.random.default_rng(0)
    d = wl.d
    n = (finite.size // d) * d
    xb = np.concatenate([rng.permutation(finite)[:n].reshape(-1, d), np.sort(finite)[:n].reshape(-1, d)])
    T = xb.shape[0]
    ids = np.sort(np.stack([np.arange(T) % wl.E, (np.arange(T) + 3) % wl.E], axis=1), axis=1).astype(np.int32)
    from block_scaled_fp4_sqrt_gb300 import MoELayer
    big = MoELayer.from_host(inp, device=device(), max_T=T, act=ACT)
    out = big.permute(x_to_device(xb), torch.from_numpy(ids).to(device()))
    torch.cuda.synchronize()
    big.check()
    counts, offsets, perm, inv = oracle.permute(ids, wl.E)
    q, s = oracle.quantize_x(xb, act=ACT)
    assert out["a_q"].shape == (T * 2, d // 2)
    assert np.array_equal(out["perm_tok"].cpu().numpy(), perm)
    assert np.array_equal(out["a_s"].cpu().numpy(), s[perm])
    assert np.array_equal(out["a_q"].cpu().numpy(), q[perm])
    big.close()


@pytest.mark.parametrize("name", ["tiny", "medium", "wide", "prefill8192"])
def test_fp4_permute_parity(name):
    wl, inp, ids_ref, wts_ref, layer = case(name, act=ACT)
    out = layer.permute(x_to_device(inp.x), torch.from_numpy(ids_ref).to(device()))
    torch.cuda.synchronize()
    layer.check()
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    q, s = oracle.quantize_x(inp.x, act=ACT)
    assert np.array_equal(out["perm_tok"].cpu().numpy(), perm)
    assert np.array_equal(out["a_q"].cpu().numpy(), q[perm])
    assert np.array_equal(out["a_s"].cpu().numpy(), s[perm])


def _forward_and_h(layer, x):
    y = layer.forward(x)
    torch.cuda.synchronize()
    layer.check()
    hq, hs = layer.last_h()
    torch.cuda.synchronize()
    return y, hq.cpu().numpy(), hs.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", None), ("tiny", 1), ("tiny", 33), ("tiny", 256), ("medium", None),
                                    ("wide", None)])
def test_fp4_forward(name, T):
    wl, inp, ids_ref, wts_ref, layer = case(name, T=T, act=ACT)
    y, hq, hs = _forward_and_h(layer, x_to_device(inp.x))
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    R = wl.T * wl.k
    assert hq.shape == (R + wl.T, wl.f // 2)
    q, s = oracle.quantize_x(inp.x, act=ACT)
    row_w = np.empty(R)
    row_w[inv.reshape(-1)] = wts_ref.reshape(-1)
    _, hq_r, hs_r, hpre_r = oracle.expert_ffn(q[perm], s[perm], inp.experts, offsets=offsets, act=ACT, want_hpre=True)
    _, hq_s, hs_s, hpre_s = oracle.expert_ffn(q, s, inp.shared, act=ACT, want_hpre=True)
    flips = check_h(hq, hs, np.concatenate([hq_r, hq_s]), np.concatenate([hs_r, hs_s]),
                    np.concatenate([hpre_r, hpre_s]), f"{name} h")
    assert flips <= max(2, hq.size // 1000)
    rows_expert = np.repeat(np.arange(wl.E), counts)
    y_ref = y_on_gpu_h(hq, hs, rows_expert, row_w, inp.experts, inp.shared, inv, wl.T, R)
    assert_close(bf16_to_f64(y), y_ref, f"{name} T={wl.T} FP4 forward")


@pytest.mark.parametrize("name", ["medium"])
def test_fp4_expert_ffn_stage(name):
    """moe_expert_ffn on the oracle's own permuted MXFP4 rows."""
    wl, inp, ids_ref, wts_ref, layer = case(name, act=ACT)
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    q, s = oracle.quantize_x(inp.x, act=ACT)
    a_q, a_s = q[perm], s[perm]
    row_w = np.empty(perm.shape[0])
    row_w[inv.reshape(-1)] = wts_ref.reshape(-1)
    dev = device()
    y = layer.expert_ffn(torch.from_numpy(a_q).to(dev), torch.from_numpy(a_s).to(dev),
                         torch.from_numpy(offsets).to(dev), torch.from_numpy(row_w.astype(np.float32)).to(dev))
    torch.cuda.synchronize()
    layer.check()
    hq, hs = (t.cpu().numpy() for t in layer.last_h())
    _, hq_r, hs_r, hpre = oracle.expert_ffn(a_q, a_s, inp.experts, offsets=offsets, act=ACT, want_hpre=True)
    check_h(hq, hs, hq_r, hs_r, hpre, f"{name} FFN h")
    rows_expert = np.repeat(np.arange(wl.E), counts)
    y_ref = np.zeros((a_q.shape[0], wl.d))
    for e in np.unique(rows_expert):
        r = np.nonzero(rows_expert == e)[0]
        y_ref[r] = oracle.down_from_h(hq[r], hs[r], inp.experts.w2[e], inp.experts.s2[e], ACT) * row_w[r, None]
    assert_close(bf16_to_f64(y), y_ref, f"{name} FP4 routed FFN")


@pytest.mark.parametrize("name", ["prefill8192", "verify512"])
def test_fp4_forward_full_size_sampled(name):
    """Full-size workloads in the benchmark's launch configuration: sampled tokens' h rows against the
    oracle, and those tokens' outputs against the oracle's down projection of the device's h."""
    wl, inp, ids_ref, wts_ref, layer = case(name, act=ACT)
    y, hq, hs = _forward_and_h(layer, x_to_device(inp.x))
    assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
    counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
    R = wl.T * wl.k
    q, s = oracle.quantize_x(inp.x, act=ACT)
    rng = np.random.default_rng(2)
    toks = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 6, replace=False)]))
    y_ref = np.zeros((toks.size, wl.d))
    for i, t in enumerate(toks):
        for j in range(wl.k):
            r, e = inv[t, j], ids_ref[t, j]
            ex = [getattr(inp.experts, n)[e] for n in ("w13", "s13", "w2", "s2")]
            _, hq_o, hs_o, hpre = oracle.expert_row(q[t], s[t], *ex, act=ACT)
            check_h(hq[r:r + 1], hs[r:r + 1], hq_o[None], hs_o[None], hpre[None], f"{name} token {t} slot {j}")
            y_ref[i] += wts_ref[t, j] * oracle.down_from_h(hq[r:r + 1], hs[r:r + 1], ex[2], ex[3], ACT)[0]
        sh = [getattr(inp.shared, n)[0] for n in ("w13", "s13", "w2", "s2")]
        _, hq_o, hs_o, hpre = oracle.expert_row(q[t], s[t], *sh, act=ACT)
        check_h(hq[R + t:R + t + 1], hs[R + t:R + t + 1], hq_o[None], hs_o[None], hpre[None], f"{name} token {t} shared")
        y_ref[i] += oracle.down_from_h(hq[R + t:R + t + 1], hs[R + t:R + t + 1], sh[2], sh[3], ACT)[0]
    assert_close(bf16_to_f64(y)[toks], y_ref, f"{name} FP4 forward (tokens {toks.tolist()})")
    y2 = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_fp4_and_fp8_layers_stay_close():
    """The variant approximates the same layer: against the MXFP8 oracle its error is that of
    activation quantisation (well above the MXFP8 path's, well below the output's size)."""
    wl, inp, ids_ref, wts_ref, layer = case("medium", act=ACT)
    y = layer.forward(x_to_device(inp.x))
    torch.cuda.synchronize()
    y8 = oracle.layer(inp.x, ids_ref, wts_ref, inp.experts, inp.shared, wl.swiglu_limit)
    rel = np.abs(bf16_to_f64(y) - y8).sum() / np.abs(y8).sum()
    assert 5e-3 < rel < 0.3


def test_shared_expert_must_match_the_format():
    from block_scaled_fp4_sqrt_gb300 import MoEError, moe_experts_set_activation_format
    wl, inp, _, _, layer = case("tiny", act=ACT)
    moe_experts_set_activation_format(layer.h_shared, "mxfp8")
    try:
        with pytest.raises(MoEError):
            layer.forward(x_to_device(inp.x))
    finally:
        moe_experts_set_activation_format(layer.h_shared, ACT)
    with pytest.raises(ValueError):
        moe_experts_set_activation_format(layer.h, "fp6")


def test_fp4_hash_layer_and_graph_replayed_stack():
    """The variant on a hash-routed layer (64 tokens, 32 experts), against the oracle on the kernel's h;
    and a two-layer stack of MXFP4 layers replayed from a CUDA graph, bit-identical to its direct launches."""
    from block_scaled_fp4_sqrt_gb300 import MoELayer, MoEStack
    wl = synth.Workload("fp4_hash", 64, 512, 256, 32, 4, hash_vocab=1000)
    inp = synth.gen_layer(wl, 4)
    ids_ref, wts_ref = oracle.hash_route(inp.token_ids, inp.hash_table, wl.k, wl.route_scale)
    layer = MoELayer.from_host(inp, device=device(), max_T=wl.T, act=ACT)
    try:
        y, hq, hs = _forward_and_h(layer, x_to_device(inp.x))
        assert np.array_equal(layer.last_topk_ids().cpu().numpy(), ids_ref)
        counts, offsets, perm, inv = oracle.permute(ids_ref, wl.E)
        R = wl.T * wl.k
        q, s = oracle.quantize_x(inp.x, act=ACT)
        _, hq_r, hs_r, hpre_r = oracle.expert_ffn(q[perm], s[perm], inp.experts, offsets=offsets, act=ACT,
                                                  want_hpre=True)
        _, hq_s, hs_s, hpre_s = oracle.expert_ffn(q, s, inp.shared, act=ACT, want_hpre=True)
        check_h(hq, hs, np.concatenate([hq_r, hq_s]), np.concatenate([hs_r, hs_s]),
                np.concatenate([hpre_r, hpre_s]), "hash FP4 h")
        row_w = np.empty(R)
        row_w[inv.reshape(-1)] = wts_ref.reshape(-1)
        y_ref = y_on_gpu_h(hq, hs, np.repeat(np.arange(wl.E), counts), row_w, inp.experts, inp.shared, inv, wl.T, R)
        assert_close(bf16_to_f64(y), y_ref, "hash FP4 forward")
        tok = layer.token_ids
        learned = synth.gen_layer(synth.Workload("fp4_learned", 64, wl.d, wl.f, wl.E, wl.k), 5)
        layer2 = MoELayer.from_host(learned, device=device(), max_T=wl.T, act=ACT, resident_router=True)
        try:
            x = x_to_device(inp.x)
            direct, graph = (MoEStack([layer, layer2], max_T=wl.T, use_graph=g) for g in (False, True))
            ref = direct.forward(x, token_ids=tok).clone()
            out = torch.empty_like(ref)
            graph.forward(x, token_ids=tok, out=out)
            graph.forward(x, token_ids=tok, out=out)
            torch.cuda.synchronize()
            graph.check()
            assert torch.equal(out, ref)
            direct.close()
            graph.close()
        finally:
            layer2.close()
    finally:
        layer.close()
