"""fp64 CPU oracle of the MoE-layer forward -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA path (``block_scaled_fp4_sqrt_gb300``); the only
thing both sides use is the seeded input generator in ``synth``.

Every function wraps one routine of ``moe_oracle.cpp`` (see its header for the passages each step
follows).  Parity status of each routine, i.e. what pins it to something other than itself, is listed
in the test modules ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

MARGIN_MIN = 1e-3  # rows whose k-th / (k+1)-th selection gap is below this are redrawn


def lib_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def _lib():
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(path)
        vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.orc_default_threads.restype = i32
        for name in ("orc_e2m1_value", "orc_e4m3_value", "orc_e8m0_value"):
            getattr(L, name).argtypes = [i32]
            getattr(L, name).restype = dbl
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_bf16_value.restype = dbl
        L.orc_mx_scale_exp.argtypes = [dbl, i32]
        L.orc_mx_scale_exp.restype = i32
        L.orc_e4m3_encode.argtypes = [dbl]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [dbl]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode_many.argtypes = [vp, i64, vp]
        L.orc_mxfp8_quantize.argtypes = [vp, i64, vp, vp]
        L.orc_mxfp4_quantize.argtypes = [vp, i64, vp, vp]
        L.orc_mxfp4_dequantize.argtypes = [vp, vp, i64, vp]
        L.orc_mxfp8_dequantize.argtypes = [vp, vp, i64, vp]
        L.orc_quantize_x.argtypes = [vp, i64, i64, vp, vp, i32, i32]
        L.orc_route.argtypes = [vp, i64, i64, vp, vp, i64, i64, dbl, i32, vp, vp, vp, vp, vp, i32]
        L.orc_hash_route.argtypes = [vp, i64, vp, i64, i64, dbl, vp, vp]
        L.orc_hash_route.restype = i64
        L.orc_permute.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.orc_expert_row.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, dbl, vp, vp, vp, vp, i32]
        L.orc_expert_ffn.argtypes = [i64, i64, vp, vp, vp, i64, i64, vp, vp, vp, vp, dbl, vp, vp, vp, vp, vp, i32,
                                     i32]
        L.orc_layer.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, dbl, vp, i64, i32,
                                vp, i32, i32]
        L.orc_layer_h.argtypes = L.orc_layer.argtypes + [vp, vp, vp]
        _LIB = L
    return _LIB


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    """Threads the oracle uses: hardware concurrency clamped by the affinity mask and the cgroup quota."""
    return int(_lib().orc_default_threads())


# ----------------------------------------------------------------------------- element formats
def e2m1_value(code: int) -> float:
    return _lib().orc_e2m1_value(int(code))


def e4m3_value(b: int) -> float:
    return _lib().orc_e4m3_value(int(b))


def e8m0_value(b: int) -> float:
    return _lib().orc_e8m0_value(int(b))


def bf16_value(h: int) -> float:
    return _lib().orc_bf16_value(int(h))


def bf16_encode(v) -> np.ndarray:
    """fp64 values -> bf16 bit patterns, round to nearest with ties to even, straight from fp64 (no
    intermediate fp32 rounding).  v = m 2^e with 0.5 <= |m| < 1; bf16 keeps 8 significant bits."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    q = np.rint(m * 256.0) / 256.0  # numpy rint rounds halves to even
    r = np.ldexp(q, e).astype(np.float32)  # exact: 8 significant bits
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def mx_blocks_unpack(blocks, split: bool):
    """17-byte MXFP4 blocks [n, 17] (E8M0 byte, then 16 bytes of 32 E2M1 codes) -> (codes [n, 16] with
    element 2i in the low nibble of byte i, scales [n]).  split: byte i of a block holds elements i (low
    nibble) and i+16 (high nibble); otherwise elements 2i and 2i+1."""
    b = np.asarray(blocks, dtype=np.uint8).reshape(-1, 17)
    q = b[:, 1:]
    if split:
        elems = np.concatenate([q & 0xF, q >> 4], axis=1)  # element e at column e
    else:
        elems = np.stack([q & 0xF, q >> 4], axis=2).reshape(-1, 32)
    codes = (elems[:, 0::2] | (elems[:, 1::2] << 4)).astype(np.uint8)
    return codes, b[:, 0].copy()


def stack_step(x_bf16, y) -> np.ndarray:
    """One layer of a stack's bf16 residual stream: x_{l+1} = bf16(x_l + y_l), the sum in fp64."""
    x = (np.asarray(x_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bf16_encode(x + np.asarray(y, dtype=np.float64))


def mx_scale_exp(amax: float, emax_elem: int) -> int:
    return _lib().orc_mx_scale_exp(float(amax), int(emax_elem))


def e4m3_encode(v) -> np.ndarray:
    v = _c(np.atleast_1d(v), np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _lib().orc_e4m3_encode_many(_p(v), v.size, _p(out))
    return out


def e2m1_encode(v: float) -> int:
    return int(_lib().orc_e2m1_encode(float(v)))


def mxfp8_quantize(v: np.ndarray):
    v = _c(v, np.float64)
    assert v.shape[-1] % 32 == 0
    q = np.empty(v.shape, dtype=np.uint8)
    s = np.empty(v.shape[:-1] + (v.shape[-1] // 32,), dtype=np.uint8)
    _lib().orc_mxfp8_quantize(_p(v), v.size, _p(q), _p(s))
    return q, s


def mxfp4_quantize(v: np.ndarray):
    v = _c(v, np.float64)
    assert v.shape[-1] % 32 == 0
    codes = np.empty(v.shape[:-1] + (v.shape[-1] // 2,), dtype=np.uint8)
    s = np.empty(v.shape[:-1] + (v.shape[-1] // 32,), dtype=np.uint8)
    _lib().orc_mxfp4_quantize(_p(v), v.size, _p(codes), _p(s))
    return codes, s


def mxfp4_dequantize(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    codes, s = _c(codes, np.uint8), _c(s, np.uint8)
    n = codes.size * 2
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.float64)
    _lib().orc_mxfp4_dequantize(_p(codes), _p(s), n, _p(out))
    return out


def mxfp8_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    out = np.empty(q.shape, dtype=np.float64)
    _lib().orc_mxfp8_dequantize(_p(q), _p(s), q.size, _p(out))
    return out


# Activation formats: "mxfp8" (the layer's: E4M3 codes, one byte per element) and "mxfp4" (the FP4
# variant: E2M1 codes, element 2i in the low nibble of byte i), one E8M0 scale per 32 elements.
ACT_FORMATS = {"mxfp8": 0, "mxfp4": 1}


def _act(act: str) -> int:
    if act not in ACT_FORMATS:
        raise ValueError(f"unknown activation format {act!r}")
    return ACT_FORMATS[act]


def act_row_bytes(act: str, n: int) -> int:
    return n // 2 if _act(act) else n


def act_dequantize(q: np.ndarray, s: np.ndarray, act: str = "mxfp8") -> np.ndarray:
    return mxfp4_dequantize(q, s) if _act(act) else mxfp8_dequantize(q, s)


def quantize_x(x_bf16: np.ndarray, act: str = "mxfp8"):
    """x bf16 [T, d] -> activation codes [T, d] (mxfp8) or [T, d/2] (mxfp4) and scales [T, d/32]."""
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    q = np.empty((T, act_row_bytes(act, d)), dtype=np.uint8)
    s = np.empty((T, d // 32), dtype=np.uint8)
    _lib().orc_quantize_x(_p(x), T, d, _p(q), _p(s), 0, _act(act))
    return q, s


# ----------------------------------------------------------------------------- routing
def route(x_bf16, router_w, router_bias, k: int, route_scale: float = 1.5, method: int = 0,
          want_logits: bool = False):
    """Returns ids int32 [T,k] (ascending), weights fp64 [T,k], margin fp64 [T] (+ logits, scores)."""
    x = _c(x_bf16, np.uint16)
    w = _c(router_w, np.float32)
    b = _c(router_bias, np.float32)
    T, d = x.shape
    E = w.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    wts = np.empty((T, k), dtype=np.float64)
    margin = np.empty((T,), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64) if want_logits else None
    scores = np.empty((T, E), dtype=np.float64) if want_logits else None
    _lib().orc_route(_p(x), T, d, _p(w), _p(b), E, k, route_scale, method, _p(ids), _p(wts), _p(margin), _p(logits),
                     _p(scores), 0)
    if want_logits:
        return ids, wts, margin, logits, scores
    return ids, wts, margin


def hash_route(token_ids, table, k: int, route_scale: float = 1.5):
    tok = _c(token_ids, np.int32)
    tab = _c(table, np.int32)
    T = tok.shape[0]
    ids = np.zeros((T, k), dtype=np.int32)
    wts = np.zeros((T, k), dtype=np.float64)
    bad = _lib().orc_hash_route(_p(tok), T, _p(tab), tab.shape[0], k, route_scale, _p(ids), _p(wts))
    if bad:
        raise ValueError(f"{bad} token ids outside the hash table")
    return ids, wts


def permute(ids, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty((E,), dtype=np.int32)
    offsets = np.empty((E + 1,), dtype=np.int32)
    perm = np.empty((T * k,), dtype=np.int32)
    inv = np.empty((T, k), dtype=np.int32)
    _lib().orc_permute(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv


# ----------------------------------------------------------------------------- experts and layer
def expert_row(aq, as_, w13, s13, w2, s2, limit: float = 10.0, act: str = "mxfp8"):
    """One expert (slices [2f, d/2], [2f, d/32], [d, f/2], [d, f/32]) on one activation row.
    Returns y fp64 [d], h codes [f] (mxfp8) or [f/2] (mxfp4), h scales [f/32], h before quantisation
    fp64 [f]."""
    aq, as_ = _c(aq, np.uint8), _c(as_, np.uint8)
    w13, s13, w2, s2 = (_c(a, np.uint8) for a in (w13, s13, w2, s2))
    d = as_.shape[-1] * 32
    f = w13.shape[0] // 2
    assert aq.shape[-1] == act_row_bytes(act, d)
    y = np.empty((d,), dtype=np.float64)
    hq = np.empty((act_row_bytes(act, f),), dtype=np.uint8)
    hs = np.empty((f // 32,), dtype=np.uint8)
    hpre = np.empty((f,), dtype=np.float64)
    _lib().orc_expert_row(_p(aq), _p(as_), d, f, _p(w13), _p(s13), _p(w2), _p(s2), limit, _p(y), _p(hq), _p(hs),
                          _p(hpre), _act(act))
    return y, hq, hs, hpre


def expert_ffn(aq, as_, weights: "synth.ExpertWeights", offsets=None, row_w=None, limit: float = 10.0,
               act: str = "mxfp8", want_hpre: bool = False):
    """Grouped FFN over activation rows (codes [n, d] for mxfp8, [n, d/2] for mxfp4; scales [n, d/32]):
    row r uses expert g with offsets[g] <= r < offsets[g+1] (offsets None: expert 0 for every row),
    scaled by row_w[r] (None: 1).  Returns y fp64 [n, d] plus the h codes and scales in the same
    format (and, with want_hpre, h before quantisation fp64 [n, f])."""
    aq, as_ = _c(aq, np.uint8), _c(as_, np.uint8)
    n = as_.shape[0]
    d = as_.shape[1] * 32
    assert aq.shape == (n, act_row_bytes(act, d))
    f = weights.w13.shape[1] // 2
    offs = None if offsets is None else _c(offsets, np.int32)
    rw = None if row_w is None else _c(row_w, np.float64)
    y = np.zeros((n, d), dtype=np.float64)
    hq = np.zeros((n, act_row_bytes(act, f)), dtype=np.uint8)
    hs = np.zeros((n, f // 32), dtype=np.uint8)
    hpre = np.zeros((n, f), dtype=np.float64) if want_hpre else None
    ng = 1 if offs is None else offs.shape[0] - 1
    _lib().orc_expert_ffn(n, ng, _p(offs), _p(aq), _p(as_), d, f, _p(_c(weights.w13, np.uint8)),
                          _p(_c(weights.s13, np.uint8)), _p(_c(weights.w2, np.uint8)), _p(_c(weights.s2, np.uint8)),
                          limit, _p(rw), _p(y), _p(hq), _p(hs), _p(hpre), 0, _act(act))
    if want_hpre:
        return y, hq, hs, hpre
    return y, hq, hs


def down_from_h(hq, hs, w2, s2, act: str = "mxfp8") -> np.ndarray:
    """The down projection of given h rows through one expert: dequantise h (codes [n, f] or packed
    [n, f/2], scales [n, f/32]) and the expert's W2 (codes [d, f/2], scales [d, f/32]) exactly, then
    one fp64 matmul.  Returns [n, d].  For checking a device path on its own h codes."""
    hd = act_dequantize(_c(hq, np.uint8), _c(hs, np.uint8), act)
    w = mxfp4_dequantize(_c(w2, np.uint8), _c(s2, np.uint8))
    return hd @ w.T


def layer(x_bf16, ids, wts, experts: "synth.ExpertWeights", shared: "synth.ExpertWeights | None",
          limit: float = 10.0, tokens=None, mode: int = 1, act: str = "mxfp8", want_h: bool = False):
    """y fp64 [n_sel, d] for the listed tokens (None: all), given the routing (ids, wts).
    mode 1 goes through the permutation; mode 0 evaluates each (token, expert) pair directly.
    act: the activation format x and h are quantised to ("mxfp8", or "mxfp4" for the FP4 variant).
    want_h: also return the h each (token, slot) row computed -- codes [n_sel, k+1, f] (or f/2 packed
    with mxfp4), scales [n_sel, k+1, f/32] and h before quantisation fp64 [n_sel, k+1, f], slot k being
    the shared expert (zeros without one) -- as (y, hq, hs, hpre)."""
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    ids = _c(ids, np.int32)
    wts = _c(wts, np.float64)
    k = ids.shape[1]
    E = experts.n
    f = experts.w13.shape[1] // 2
    tok = None if tokens is None else _c(tokens, np.int32)
    n_sel = T if tok is None else tok.shape[0]
    y = np.empty((n_sel, d), dtype=np.float64)
    sh = [None] * 4 if shared is None else [_c(a, np.uint8) for a in (shared.w13, shared.s13, shared.w2, shared.s2)]
    ex = [_c(a, np.uint8) for a in (experts.w13, experts.s13, experts.w2, experts.s2)]
    if not want_h:
        _lib().orc_layer(_p(x), T, d, f, E, k, _p(ids), _p(wts), *(_p(a) for a in ex), *(_p(a) for a in sh), limit,
                         _p(tok), n_sel, mode, _p(y), 0, _act(act))
        return y
    hq = np.zeros((n_sel, k + 1, act_row_bytes(act, f)), dtype=np.uint8)
    hs = np.zeros((n_sel, k + 1, f // 32), dtype=np.uint8)
    hpre = np.zeros((n_sel, k + 1, f), dtype=np.float64)
    _lib().orc_layer_h(_p(x), T, d, f, E, k, _p(ids), _p(wts), *(_p(a) for a in ex), *(_p(a) for a in sh), limit,
                       _p(tok), n_sel, mode, _p(y), 0, _act(act), _p(hq), _p(hs), _p(hpre))
    return y, hq, hs, hpre


def route_inputs(inp: "synth.LayerInputs"):
    """Routing of a generated layer: (ids, wts, margin-or-None)."""
    wl = inp.wl
    if wl.hashed:
        ids, wts = hash_route(inp.token_ids, inp.hash_table, wl.k, wl.route_scale)
        return ids, wts, None
    return route(inp.x, inp.router_w, inp.router_bias, wl.k, wl.route_scale)


def margin_filtered_layer(wl: "synth.Workload", seed: int = 0, threshold: float = MARGIN_MIN,
                          with_shared: bool = True, adjust=None, x_scale: float = 1.0):
    """Generate a layer and redraw (per row, up to 255 times) every x row whose top-k selection gap is
    below ``threshold``, so that the selection does not depend on the precision it is computed in.
    ``adjust(inputs)`` may edit the generated inputs (e.g. the router bias) before routing; x rows are
    drawn with standard deviation ``x_scale``.  Returns (inputs, ids, wts, margin)."""
    inp = synth.gen_layer(wl, seed, with_shared=with_shared)
    if x_scale != 1.0:
        inp.x = synth.gen_x(seed, wl.T, wl.d, scale=x_scale)
    if adjust is not None:
        adjust(inp)
    ids, wts, margin = route_inputs(inp)
    if wl.hashed:
        return inp, ids, wts, margin
    attempts = np.zeros((wl.T,), dtype=np.int32)
    for _ in range(255):
        low = np.nonzero(margin < threshold)[0]
        if low.size == 0:
            break
        attempts[low] += 1
        xs = synth.gen_x(seed, wl.T, wl.d, attempts, scale=x_scale)
        inp.x[low] = xs[low]
        ids_l, wts_l, m_l = route(inp.x[low], inp.router_w, inp.router_bias, wl.k, wl.route_scale)
        ids[low], wts[low], margin[low] = ids_l, wts_l, m_l
    else:
        raise RuntimeError("margin rejection did not converge")
    inp.attempts = attempts
    return inp, ids, wts, margin
