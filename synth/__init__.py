"""Seeded synthetic workloads for the MoE-layer forward.

This module only draws inputs: x, the router weight and bias, MXFP4 expert weights, token ids and
the hash table.  It holds none of the layer's arithmetic and is shared by the oracle side and the
CUDA side.  The native part (``libsynth.so``) is compiled by ``__graft_entry__.build()``.

Workloads (one per row of the benchmark table):

==============  =====  =====  =====  ===  =  =====================================================
name            T      d      f      E    k  notes
==============  =====  =====  =====  ===  =  =====================================================
tiny            16     256    128    8    2  small layer for element-wise parity
verify512       512    4096   2048   256  6  64 requests x 8 verify rows (1 + 7 drafts)
verify8         8      4096   2048   256  6  one request's verify rows; weight-bandwidth bound
hash512         512    4096   2048   256  6  hash-routed layer: token id -> table of 6 expert ids
prefill8192     8192   4096   2048   256  6  prefill chunk, 26 hot experts get router bias +1.0
==============  =====  =====  =====  ===  =  =====================================================

All have one shared expert with the routed experts' FFN width, route scale 1.5, SwiGLU limit 10.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, "libsynth.so")


def _lib():
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(path)
        u64, i64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.synth_x_bf16.argtypes = [u64, i64, i64, dbl, vp, vp, i32]
        L.synth_router.argtypes = [u64, i64, i64, vp, vp]
        L.synth_hot_bias.argtypes = [u64, i64, i64, ctypes.c_float, vp, vp]
        L.synth_mxfp4.argtypes = [u64, i32, i32, i64, i64, i64, i64, vp, vp, i32]
        L.synth_token_ids.argtypes = [u64, i64, i64, vp]
        L.synth_hash_table.argtypes = [u64, i64, i64, i64, vp]
        L.synth_u64.argtypes = [u64, u64, u64]
        L.synth_u64.restype = ctypes.c_uint64
        L.synth_normal.argtypes = [u64, u64, u64]
        L.synth_normal.restype = ctypes.c_double
        L.synth_weight_e0.argtypes = [i64]
        L.synth_weight_e0.restype = ctypes.c_int
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    route_scale: float = 1.5
    swiglu_limit: float = 10.0
    hash_vocab: int = 0          # > 0: hash-routed layer with this many token ids
    n_hot: int = 0               # experts given +hot_bias on the router bias
    hot_bias: float = 1.0
    description: str = field(default="", compare=False)

    @property
    def hashed(self) -> bool:
        return self.hash_vocab > 0

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_T(self, T: int) -> "Workload":
        return Workload(self.name, T, self.d, self.f, self.E, self.k, self.route_scale, self.swiglu_limit,
                        self.hash_vocab, self.n_hot, self.hot_bias, self.description)


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 128, 8, 2, description="T=16, d=256, f=128, 8 experts top-2 + 1 shared"),
    "verify512": Workload("verify512", 512, 4096, 2048, 256, 6,
                          description="T=512 verify rows (64 requests x 8), d=4096, f=2048, 256 experts top-6 + 1 shared"),
    "verify8": Workload("verify8", 8, 4096, 2048, 256, 6,
                        description="T=8 verify rows (1 request x 8), d=4096, f=2048, 256 experts top-6 + 1 shared"),
    "hash512": Workload("hash512", 512, 4096, 2048, 256, 6, hash_vocab=131072,
                        description="T=512 hash-routed, token ids ~U[0,131072), table 131072x6"),
    "prefill8192": Workload("prefill8192", 8192, 4096, 2048, 256, 6, n_hot=26, hot_bias=1.0,
                            description="T=8192 prefill chunk, 26 of 256 experts get router bias +1.0"),
}


def gen_x(seed: int, T: int, d: int, attempts: np.ndarray | None = None, scale: float = 1.0,
          threads: int | None = None) -> np.ndarray:
    """x rows as bf16 bit patterns (uint16 [T, d]); ``attempts[t]`` redraws row t independently."""
    out = np.empty((T, d), dtype=np.uint16)
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.int32)
        if att.shape != (T,) or att.min(initial=0) < 0 or att.max(initial=0) > 255:
            raise ValueError("attempts must be int32 [T] in 0..255")
    _lib().synth_x_bf16(seed, T, d, scale, _ptr(att), _ptr(out), threads or default_threads())
    return out


def gen_router(seed: int, E: int, d: int, n_hot: int = 0, hot_bias: float = 1.0):
    """Router weight fp32 [E, d] ~ N(0, 1/d), bias fp32 [E] ~ U(-0.1, 0.1) (+hot_bias on n_hot experts)."""
    w = np.empty((E, d), dtype=np.float32)
    b = np.empty((E,), dtype=np.float32)
    _lib().synth_router(seed, E, d, _ptr(w), _ptr(b))
    hot = np.empty((max(n_hot, 0),), dtype=np.int32)
    if n_hot > 0:
        _lib().synth_hot_bias(seed, E, n_hot, hot_bias, _ptr(b), _ptr(hot))
    return w, b, hot


def gen_mxfp4(seed: int, stream_codes: int, stream_scales: int, rows: int, cols: int, d_in: int,
              row0: int = 0, threads: int | None = None):
    codes = np.empty((rows, cols // 2), dtype=np.uint8)
    scales = np.empty((rows, cols // 32), dtype=np.uint8)
    _lib().synth_mxfp4(seed, stream_codes, stream_scales, row0, rows, cols, d_in, _ptr(codes), _ptr(scales),
                       threads or default_threads())
    return codes, scales


@dataclass
class ExpertWeights:
    """Canonical MXFP4 expert set: gate-up rows [n, 2f, d] (rows 0..f-1 gate, f..2f-1 up) and down
    rows [n, d, f]; codes hold element 2i in the low nibble of byte i, scales are E8M0 bytes."""
    w13: np.ndarray      # uint8 [n, 2f, d/2]
    s13: np.ndarray      # uint8 [n, 2f, d/32]
    w2: np.ndarray       # uint8 [n, d, f/2]
    s2: np.ndarray       # uint8 [n, d, f/32]

    @property
    def n(self) -> int:
        return self.w13.shape[0]


def gen_experts(seed: int, n: int, d: int, f: int, shared: bool = False, threads: int | None = None) -> ExpertWeights:
    sc13, ss13, sc2, ss2 = (5, 10, 13, 14) if shared else (4, 9, 11, 12)
    w13, s13 = gen_mxfp4(seed, sc13, ss13, n * 2 * f, d, d, threads=threads)
    w2, s2 = gen_mxfp4(seed, sc2, ss2, n * d, f, d, threads=threads)
    return ExpertWeights(w13.reshape(n, 2 * f, d // 2), s13.reshape(n, 2 * f, d // 32),
                         w2.reshape(n, d, f // 2), s2.reshape(n, d, f // 32))


def gen_token_ids(seed: int, T: int, V: int) -> np.ndarray:
    tok = np.empty((T,), dtype=np.int32)
    _lib().synth_token_ids(seed, T, V, _ptr(tok))
    return tok


def gen_hash_table(seed: int, V: int, E: int, k: int) -> np.ndarray:
    tab = np.empty((V, k), dtype=np.int32)
    _lib().synth_hash_table(seed, V, E, k, _ptr(tab))
    return tab


@dataclass
class LayerInputs:
    wl: Workload
    seed: int
    x: np.ndarray                    # uint16 bf16 bits [T, d]
    router_w: np.ndarray | None      # fp32 [E, d]
    router_bias: np.ndarray | None   # fp32 [E]
    experts: ExpertWeights
    shared: ExpertWeights | None
    token_ids: np.ndarray | None     # int32 [T] (hash layers)
    hash_table: np.ndarray | None    # int32 [V, k] (hash layers)
    hot_ids: np.ndarray | None = None
    attempts: np.ndarray | None = None


def gen_layer(wl: Workload, seed: int = 0, attempts: np.ndarray | None = None, with_shared: bool = True,
              threads: int | None = None, experts: ExpertWeights | None = None) -> LayerInputs:
    """All inputs of one layer forward.  The router (or hash table) is drawn even when a test later
    replaces x rows through ``attempts``; weights never depend on x.  ``experts``: routed weights already
    drawn for the same (seed, E, d, f), which are then reused instead of drawn again."""
    x = gen_x(seed, wl.T, wl.d, attempts, threads=threads)
    if experts is None:
        experts = gen_experts(seed, wl.E, wl.d, wl.f, shared=False, threads=threads)
    elif experts.w13.shape != (wl.E, 2 * wl.f, wl.d // 2):
        raise ValueError("reused expert weights do not match the workload's shape")
    shared = gen_experts(seed, 1, wl.d, wl.f, shared=True, threads=threads) if with_shared else None
    if wl.hashed:
        tok = gen_token_ids(seed, wl.T, wl.hash_vocab)
        tab = gen_hash_table(seed, wl.hash_vocab, wl.E, wl.k)
        return LayerInputs(wl, seed, x, None, None, experts, shared, tok, tab, None, attempts)
    w, b, hot = gen_router(seed, wl.E, wl.d, wl.n_hot, wl.hot_bias)
    return LayerInputs(wl, seed, x, w, b, experts, shared, None, None, hot if wl.n_hot else None, attempts)
