"""Shared set-up of the GPU parity tests: seeded, margin-filtered layers on the device next to the
oracle's routing, and the parity tolerances."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth

# Layer output (floating point), from the layer's contract: max |y - y_ref| <= 2e-2 rms(y_ref) and
# sum |y - y_ref| / sum |y_ref| <= 5e-3.
TOL_MAX_RMS = 2e-2
TOL_MEAN_REL = 5e-3
# Routing weights: fp32 logits are dot products of length d; their error is a few units of
# 2^-24 * sqrt(d) * sum_i |x_i w_i| (~1e-5 of the score for d = 4096), so 1e-4 relative bounds the
# weights with margin.
TOL_WEIGHT_REL = 1e-4

# A mid-size layer that the oracle evaluates in seconds but that still spans several output tiles
# (f/128 = 4 gate-up, d/128 = 8 down), several K stages per tile, more work items than SMs and
# expert groups longer than one 32-row tile.
MEDIUM = synth.Workload("medium", 512, 1024, 512, 16, 4, description="T=512, d=1024, f=512, 16 experts top-4")

# More routed experts than one 256-wide router tile: the learned router's two-kernel path (logits, then a
# separate split-K reduction with top-k over two expert tiles) instead of the fused cluster router.
WIDE = synth.Workload("wide", 96, 512, 128, 384, 6, description="T=96, d=512, f=128, 384 experts top-6")

WORKLOADS = dict(synth.WORKLOADS, medium=MEDIUM, wide=WIDE)


def device():
    return torch.device("cuda:0")


def x_to_device(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(device()).view(torch.bfloat16)


@functools.lru_cache(maxsize=1)
def case(name: str, T: int | None = None, seed: int = 0, act: str = "mxfp8"):
    """(workload, inputs, oracle ids, oracle weights, device layer) for a named workload; act is the
    layer's activation format ("mxfp4": the MXFP4-activation variant)."""
    from block_scaled_fp4_sqrt_gb300 import MoELayer
    wl = WORKLOADS[name]
    if T is not None:
        wl = wl.with_T(T)
    inp, ids, wts, _ = oracle.margin_filtered_layer(wl, seed)
    layer = MoELayer.from_host(inp, device=device(), max_T=max(wl.T, 1), act=act)
    return wl, inp, ids, wts, layer


def compare_outputs(y: np.ndarray, y_ref: np.ndarray):
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    max_err = float(np.max(np.abs(y - y_ref))) if y.size else 0.0
    mean_rel = float(np.sum(np.abs(y - y_ref)) / max(np.sum(np.abs(y_ref)), 1e-300)) if y.size else 0.0
    return max_err, rms, mean_rel


# The outputs compared here are bf16: each element carries one rounding to bf16 (8 significant bits,
# at most 2^-8 of its magnitude) on top of the arithmetic the tolerance above bounds.  A layer output
# of 2M elements reaches 7 rms in its tail, where that rounding alone is 2.7e-2 rms; so the
# element-wise bound is TOL_MAX_RMS * rms + 2^-8 |y_ref|.
BF16_HALF_ULP_REL = 2.0 ** -8


def assert_close(y: np.ndarray, y_ref: np.ndarray, what: str = "output"):
    """For outputs that exist only in bf16 (the grouped FFN call's rows, a stack's residual stream): the
    contract's bound plus the output's own rounding.  The strict figure is printed beside it."""
    max_err, rms, mean_rel = compare_outputs(y, y_ref)
    print(f"{what}: max |dy| / rms = {max_err / max(rms, 1e-300):.4e} (bf16 output; strict bound "
          f"{TOL_MAX_RMS} applies before the rounding), mean rel = {mean_rel:.4e}")
    excess = np.abs(y - y_ref) - (TOL_MAX_RMS * rms + BF16_HALF_ULP_REL * np.abs(y_ref)) if y.size else np.zeros(1)
    assert np.all(excess <= 0), (f"{what}: max |dy| {max_err:.4e} exceeds {TOL_MAX_RMS} rms ({rms:.4e}) plus the bf16 "
                                 f"rounding of y_ref by {float(excess.max()):.4e}")
    assert mean_rel <= TOL_MEAN_REL, f"{what}: mean relative error {mean_rel:.4e} > {TOL_MEAN_REL}"
    return max_err / max(rms, 1e-300), mean_rel


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_strict(y32: np.ndarray, y_ref: np.ndarray, what: str = "output"):
    """The layer's contract as written, on the fp32 sums before the output's rounding to bf16:
    max |y - y_ref| <= 2e-2 rms(y_ref) and sum |y - y_ref| / sum |y_ref| <= 5e-3, nothing added."""
    max_err, rms, mean_rel = compare_outputs(y32, y_ref)
    print(f"{what}: strict max |dy| / rms = {max_err / max(rms, 1e-300):.4e} (bound {TOL_MAX_RMS}), "
          f"mean rel = {mean_rel:.4e} (bound {TOL_MEAN_REL})")
    assert max_err <= TOL_MAX_RMS * rms, f"{what}: max |dy| {max_err:.4e} > {TOL_MAX_RMS} rms ({rms:.4e})"
    assert mean_rel <= TOL_MEAN_REL, f"{what}: mean relative error {mean_rel:.4e} > {TOL_MEAN_REL}"
    return max_err / max(rms, 1e-300), mean_rel


def assert_bf16_is_rne_of(y_bf16: torch.Tensor, y32: torch.Tensor, what: str = "output"):
    """The bf16 output is the fp32 sum rounded once to nearest even, bit for bit (torch's fp32 -> bf16
    conversion rounds to nearest even)."""
    want = y32.to(torch.bfloat16).view(torch.int16)
    got = y_bf16.view(torch.int16)
    n_bad = int((want != got).sum().item())
    assert n_bad == 0, f"{what}: {n_bad} bf16 outputs are not the round-to-nearest-even of their fp32 sums"


def forward_strict(layer, x: torch.Tensor, token_ids=None):
    """moe_forward, then its bf16 output and the fp32 sums it was rounded from (checked to agree)."""
    y = layer.forward(x, token_ids=token_ids)
    y32 = layer.last_y32()
    torch.cuda.synchronize()
    layer.check()
    assert_bf16_is_rne_of(y, y32)
    return y, y32


# E4M3 magnitudes (subnormals m 2^-9, normals (1 + m/8) 2^(e-7), largest 448) and the midpoints where
# round-to-nearest-even changes code.
_E4M3 = np.array(sorted({m * 2.0 ** -9 for m in range(8)} |
                        {(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8) if (e, m) != (15, 7)}))
E4M3_MIDPOINTS = (_E4M3[1:] + _E4M3[:-1]) / 2


def _e4m3_fragile(hpre: np.ndarray, hs_ref: np.ndarray):
    """(code_fragile [n, f], scale_fragile [n, f/32]) of MXFP8 h from the oracle's h before quantisation.
    The kernels' h is an fp32 sum of exact products: a few 1e-6 of the largest partial sum, which in
    units of the block scale (2^-8 of the block maximum and below) is up to a few 2^-10.  A code may
    therefore differ where the oracle's value lies within 2^-10 relative plus 2^-8 absolute (block
    units) of a rounding midpoint; a scale byte where the block maximum is within 1.5e-4 of a power of two."""
    n, f = hpre.shape
    blocks = hpre.reshape(n, f // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    scale_fragile = (amax > 0) & (np.abs(lg - np.round(lg)) <= 1.5e-4)
    unit = np.ldexp(1.0, hs_ref.astype(np.int64) - 127)[:, :, None]
    v = (np.abs(blocks) / unit).reshape(n, f)
    idx = np.clip(np.searchsorted(E4M3_MIDPOINTS, v), 1, E4M3_MIDPOINTS.size - 1)
    dist = np.minimum(np.abs(v - E4M3_MIDPOINTS[idx - 1]), np.abs(v - E4M3_MIDPOINTS[idx]))
    return dist <= 2.0 ** -10 * v + 2.0 ** -8, scale_fragile


def check_h8(hq_gpu, hs_gpu, hq_ref, hs_ref, hpre, what):
    """MXFP8 h codes and scales equal the oracle's except where the oracle's own h is fragile (above);
    a code that is zero in magnitude on both sides may differ in its sign bit only.  At most 0.1 % of
    the codes may differ.  Returns the number of differing codes (32 per differing scale)."""
    hq_gpu, hs_gpu, hq_ref, hs_ref = (np.asarray(a) for a in (hq_gpu, hs_gpu, hq_ref, hs_ref))
    code_fragile, scale_fragile = _e4m3_fragile(np.asarray(hpre), hs_ref)
    bad_scale = hs_gpu != hs_ref
    assert not np.any(bad_scale & ~scale_fragile), \
        f"{what}: {int(np.sum(bad_scale & ~scale_fragile))} h scale bytes differ outside fragile blocks"
    same_scale = np.repeat(~bad_scale, 32, axis=1)
    both_zero = ((hq_gpu & 0x7F) == 0) & ((hq_ref & 0x7F) == 0)
    bad_code = (hq_gpu != hq_ref) & same_scale & ~both_zero
    n_hard = int(np.sum(bad_code & ~code_fragile))
    assert n_hard == 0, f"{what}: {n_hard} h codes differ away from a rounding midpoint"
    flips = int(bad_code.sum()) + 32 * int(bad_scale.sum())
    print(f"{what}: {flips} of {hq_gpu.size} h codes at fragile midpoints differ")
    assert flips <= max(2, hq_gpu.size // 1000), f"{what}: {flips} h codes differ"
    return flips


def gpu_h_by_slot(hq_dev: np.ndarray, hs_dev: np.ndarray, inv: np.ndarray, tokens: np.ndarray, R: int,
                  has_shared: bool = True):
    """The device's h rows (routed rows in permuted order, then one shared row per token) rearranged to
    the oracle's [n_sel, k + 1, ...] order for the given tokens (slot k: the shared row)."""
    k = inv.shape[1]
    rows = np.concatenate([inv[tokens], (R + tokens)[:, None]], axis=1) if has_shared else inv[tokens]
    return hq_dev[rows], hs_dev[rows]
