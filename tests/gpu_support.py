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
    max_err, rms, mean_rel = compare_outputs(y, y_ref)
    excess = np.abs(y - y_ref) - (TOL_MAX_RMS * rms + BF16_HALF_ULP_REL * np.abs(y_ref)) if y.size else np.zeros(1)
    assert np.all(excess <= 0), (f"{what}: max |dy| {max_err:.4e} exceeds {TOL_MAX_RMS} rms ({rms:.4e}) plus the bf16 "
                                 f"rounding of y_ref by {float(excess.max()):.4e}")
    assert mean_rel <= TOL_MEAN_REL, f"{what}: mean relative error {mean_rel:.4e} > {TOL_MEAN_REL}"
    return max_err / max(rms, 1e-300), mean_rel


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
