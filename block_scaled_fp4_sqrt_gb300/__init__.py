"""GB300-native forward pass of a DeepSeek-V4-Flash-style MoE layer (sqrt-softplus router, MXFP4
experts, SwiGLU with clamp, weighted combine) -- Python binding of ``libmoe.so``.

The functions below carry the C-ABI names of ``include/moe.h`` and only marshal arguments: every
step of the layer runs in the library's sm_103a kernels.  PyTorch provides device memory and
streams.  There is no fallback: importing works anywhere, but every call raises if ``libmoe.so`` is
missing or cannot be loaded.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
_LIB = None

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_CHECK", 6: "MOE_ERR_TIMEOUT"}

EXPORTED = ("moe_experts_create", "moe_experts_set_hash_table", "moe_workspace_size", "moe_set_workspace",
            "moe_route", "moe_permute", "moe_expert_ffn", "moe_forward", "moe_get_routing", "moe_check",
            "moe_set_wait_budget", "moe_experts_destroy", "moe_status_string", "moe_last_error",
            "moe_testing_stall_loads", "moe_set_stage_events", "moe_route_noalloc", "moe_measure_mxf8f6f4_peak",
            "moe_stack_create", "moe_stack_forward", "moe_stack_destroy", "moe_mx_blocks_unpack",
            "moe_experts_set_activation_format", "moe_measure_mxf4_peak", "moe_testing_read_h",
            "moe_experts_set_router", "moe_testing_read_y32", "moe_testing_set_pair_gemm")

MOE_MX_NIBBLES_PAIRED, MOE_MX_NIBBLES_SPLIT = 0, 1
MOE_ACT_MXFP8, MOE_ACT_MXFP4 = 0, 1
ACT_FORMATS = {"mxfp8": MOE_ACT_MXFP8, "mxfp4": MOE_ACT_MXFP4}

MOE_N_STAGES = 5
STAGE_NAMES = ("route", "dispatch", "gemm_gate_up", "gemm_down", "combine")


class MoEError(RuntimeError):
    def __init__(self, call: str, status: int, message: str):
        super().__init__(f"{call}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class moe_config_t(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("route_scale", ctypes.c_float), ("swiglu_limit", ctypes.c_float)]


class moe_stack_layer_t(ctypes.Structure):
    _fields_ = [("experts", ctypes.c_void_p), ("shared", ctypes.c_void_p), ("router_w", ctypes.c_void_p),
                ("router_bias", ctypes.c_void_p)]


class moe_input_t(ctypes.Structure):
    _fields_ = [("x_bf16", ctypes.c_void_p), ("T", ctypes.c_int32), ("token_ids", ctypes.c_void_p)]


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int
        cfgp, inp = ctypes.POINTER(moe_config_t), ctypes.POINTER(moe_input_t)
        L.moe_experts_create.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, ctypes.POINTER(vp)]
        L.moe_experts_set_hash_table.argtypes = [vp, vp, i32]
        L.moe_workspace_size.argtypes = [cfgp, i32]
        L.moe_workspace_size.restype = ctypes.c_size_t
        L.moe_set_workspace.argtypes = [vp, vp, ctypes.c_size_t, i32]
        L.moe_route.argtypes = [vp, inp, vp, vp, vp, vp, vp]
        L.moe_permute.argtypes = [vp, inp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_expert_ffn.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_forward.argtypes = [inp, vp, vp, vp, vp, vp, vp]
        L.moe_get_routing.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i32)]
        L.moe_check.argtypes = [vp, vp]
        L.moe_set_wait_budget.argtypes = [vp, u64]
        L.moe_testing_stall_loads.argtypes = [vp, i32]
        L.moe_set_stage_events.argtypes = [vp, ctypes.POINTER(vp), i32]
        L.moe_route_noalloc.argtypes = [cfgp, inp, vp, vp, vp, vp, vp]
        L.moe_measure_mxf8f6f4_peak.argtypes = [i32, ctypes.POINTER(ctypes.c_double)]
        L.moe_measure_mxf4_peak.argtypes = [i32, ctypes.POINTER(ctypes.c_double)]
        L.moe_experts_set_activation_format.argtypes = [vp, i32]
        L.moe_testing_read_h.argtypes = [vp, vp, vp, ctypes.POINTER(i32), vp]
        L.moe_experts_set_router.argtypes = [vp, vp, vp, vp]
        L.moe_testing_read_y32.argtypes = [vp, vp, ctypes.POINTER(i32), vp]
        L.moe_testing_set_pair_gemm.argtypes = [vp, i32]
        L.moe_stack_create.argtypes = [ctypes.POINTER(moe_stack_layer_t), i32, i32, ctypes.POINTER(vp)]
        L.moe_stack_forward.argtypes = [vp, inp, vp, vp, vp]
        L.moe_stack_destroy.argtypes = [vp]
        L.moe_mx_blocks_unpack.argtypes = [vp, ctypes.c_int64, i32, vp, vp, vp]
        L.moe_stack_destroy.restype = None
        L.moe_experts_destroy.argtypes = [vp]
        L.moe_experts_destroy.restype = None
        L.moe_status_string.argtypes = [st]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("moe_workspace_size", "moe_experts_destroy", "moe_status_string", "moe_last_error",
                            "moe_stack_destroy"):
                getattr(L, name).restype = st
        _LIB = L
    return _LIB


def _ok(call: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(call, status, lib().moe_last_error().decode())


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _input(x: torch.Tensor, token_ids: torch.Tensor | None = None) -> moe_input_t:
    return moe_input_t(ctypes.c_void_p(x.data_ptr()) if x.numel() else None, int(x.shape[0]),
                       None if token_ids is None else ctypes.c_void_p(token_ids.data_ptr()))


def make_config(d_model: int, d_ff: int, n_experts: int, top_k: int, route_scale: float = 1.5,
                swiglu_limit: float = 10.0) -> moe_config_t:
    return moe_config_t(d_model, d_ff, n_experts, top_k, route_scale, swiglu_limit)


# ----------------------------------------------------------------------------- C-ABI wrappers
def moe_experts_create(cfg: moe_config_t, n: int, w13: torch.Tensor, s13: torch.Tensor, w2: torch.Tensor,
                       s2: torch.Tensor, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _ok("moe_experts_create", lib().moe_experts_create(ctypes.byref(cfg), n, _p(w13), _p(s13), _p(w2), _p(s2),
                                                       _stream(stream), ctypes.byref(h)))
    return h


def moe_experts_set_hash_table(h, table: torch.Tensor | None) -> None:
    _ok("moe_experts_set_hash_table",
        lib().moe_experts_set_hash_table(h, _p(table), 0 if table is None else int(table.shape[0])))


def moe_experts_set_router(h, router_w: torch.Tensor | None, router_bias: torch.Tensor | None, stream=None) -> None:
    _ok("moe_experts_set_router", lib().moe_experts_set_router(h, _p(router_w), _p(router_bias), _stream(stream)))


def moe_workspace_size(cfg: moe_config_t, max_T: int) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg), max_T))


def moe_set_workspace(h, ws: torch.Tensor, max_T: int) -> None:
    _ok("moe_set_workspace", lib().moe_set_workspace(h, _p(ws), ws.numel() * ws.element_size(), max_T))


def moe_route(h, x, router_w, router_bias, topk_ids, topk_w, token_ids=None, stream=None) -> None:
    _ok("moe_route", lib().moe_route(h, ctypes.byref(_input(x, token_ids)), _p(router_w), _p(router_bias),
                                     _p(topk_ids), _p(topk_w), _stream(stream)))


def moe_permute(h, x, topk_ids, counts, offsets, perm_tok, inv_pos, a_q=None, a_s=None, stream=None) -> None:
    _ok("moe_permute", lib().moe_permute(h, ctypes.byref(_input(x)), _p(topk_ids), _p(counts), _p(offsets),
                                         _p(perm_tok), _p(inv_pos), _p(a_q), _p(a_s), _stream(stream)))


def moe_expert_ffn(h, n_rows: int, offsets, a_q, a_s, row_w, y, stream=None) -> None:
    _ok("moe_expert_ffn", lib().moe_expert_ffn(h, n_rows, _p(offsets), _p(a_q), _p(a_s), _p(row_w), _p(y),
                                               _stream(stream)))


def moe_forward(x, router_w, router_bias, experts, shared, out, token_ids=None, stream=None) -> None:
    _ok("moe_forward", lib().moe_forward(ctypes.byref(_input(x, token_ids)), _p(router_w), _p(router_bias),
                                         experts, shared, _p(out), _stream(stream)))


def moe_get_routing(h):
    ids, w, T = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int32()
    _ok("moe_get_routing", lib().moe_get_routing(h, ctypes.byref(ids), ctypes.byref(w), ctypes.byref(T)))
    return ids.value, w.value, T.value


def moe_check(h, stream=None) -> None:
    _ok("moe_check", lib().moe_check(h, _stream(stream)))


def moe_set_wait_budget(h, budget_ns: int) -> None:
    _ok("moe_set_wait_budget", lib().moe_set_wait_budget(h, budget_ns))


def moe_testing_stall_loads(h, enable: bool) -> None:
    _ok("moe_testing_stall_loads", lib().moe_testing_stall_loads(h, 1 if enable else 0))


def moe_measure_mxf8f6f4_peak(n_stages: int = 4096) -> float:
    """Measured dense TFLOP/s of the block-scaled E4M3 x E2M1 MMA (M=128, N=256, K=32) on the
    current device; synchronous."""
    out = ctypes.c_double(0.0)
    _ok("moe_measure_mxf8f6f4_peak", lib().moe_measure_mxf8f6f4_peak(int(n_stages), ctypes.byref(out)))
    return out.value


def moe_measure_mxf4_peak(n_stages: int = 4096) -> float:
    """Measured dense TFLOP/s of the block-scaled E2M1 x E2M1 MMA (kind::mxf4, M=128, N=256, K=64) on
    the current device; synchronous."""
    out = ctypes.c_double(0.0)
    _ok("moe_measure_mxf4_peak", lib().moe_measure_mxf4_peak(int(n_stages), ctypes.byref(out)))
    return out.value


def moe_testing_read_h(h, f: int, act: str, stream=None):
    """The h codes and canonical scales of the last grouped FFN on the handle (device tensors)."""
    n = ctypes.c_int32(0)
    _ok("moe_testing_read_h", lib().moe_testing_read_h(h, None, None, ctypes.byref(n), _stream(stream)))
    dev = torch.device("cuda", torch.cuda.current_device())
    hq = torch.empty((n.value, f // 2 if act == "mxfp4" else f), dtype=torch.uint8, device=dev)
    hs = torch.empty((n.value, f // 32), dtype=torch.uint8, device=dev)
    if n.value:
        _ok("moe_testing_read_h", lib().moe_testing_read_h(h, _p(hq), _p(hs), ctypes.byref(n), _stream(stream)))
    return hq, hs


def moe_testing_set_pair_gemm(h, enable: bool) -> None:
    """Run 128-row tiles on the CTA-pair GEMMs, or on the one-SM kernels (the default)."""
    _ok("moe_testing_set_pair_gemm", lib().moe_testing_set_pair_gemm(h, 1 if enable else 0))


def moe_testing_read_y32(h, d: int, stream=None) -> torch.Tensor:
    """The fp32 sums of the last moe_forward on the handle before their rounding to bf16 ([T, d])."""
    n = ctypes.c_int32(0)
    _ok("moe_testing_read_y32", lib().moe_testing_read_y32(h, None, ctypes.byref(n), _stream(stream)))
    dev = torch.device("cuda", torch.cuda.current_device())
    y = torch.empty((n.value, d), dtype=torch.float32, device=dev)
    if n.value:
        _ok("moe_testing_read_y32", lib().moe_testing_read_y32(h, _p(y), ctypes.byref(n), _stream(stream)))
    return y


def moe_experts_set_activation_format(h, fmt: str) -> None:
    """fmt: "mxfp8" (the layer's) or "mxfp4" (the MXFP4-activation variant)."""
    if fmt not in ACT_FORMATS:
        raise ValueError(f"unknown activation format {fmt!r}")
    _ok("moe_experts_set_activation_format", lib().moe_experts_set_activation_format(h, ACT_FORMATS[fmt]))


def moe_set_stage_events(h, events) -> object:
    """events: MOE_N_STAGES + 1 torch.cuda.Event(enable_timing=True) (or None to stop).  Returns the
    ctypes array the library reads; keep it alive while recording."""
    if events is None:
        _ok("moe_set_stage_events", lib().moe_set_stage_events(h, None, 0))
        return None
    for e in events:  # torch creates the underlying event on first record
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _ok("moe_set_stage_events", lib().moe_set_stage_events(h, arr, len(events)))
    return arr


def moe_route_noalloc(cfg: moe_config_t, x, router_w, router_bias, topk_ids, topk_w, stream=None) -> None:
    """Learned router without a handle or workspace (fixed library scratch; see include/moe.h)."""
    _ok("moe_route_noalloc", lib().moe_route_noalloc(ctypes.byref(cfg), ctypes.byref(_input(x)), _p(router_w),
                                                     _p(router_bias), _p(topk_ids), _p(topk_w), _stream(stream)))


def moe_stack_create(layers, use_graph: bool):
    """layers: sequence of (experts handle, shared handle or None, router_w or None, router_bias or None)."""
    arr = (moe_stack_layer_t * len(layers))()
    for i, (h, sh, rw, rb) in enumerate(layers):
        arr[i] = moe_stack_layer_t(h, sh, None if rw is None else rw.data_ptr(), None if rb is None else rb.data_ptr())
    out = ctypes.c_void_p()
    _ok("moe_stack_create", lib().moe_stack_create(arr, len(layers), 1 if use_graph else 0, ctypes.byref(out)))
    return out


def moe_stack_forward(stack, x, out, scratch, token_ids=None, stream=None) -> None:
    _ok("moe_stack_forward", lib().moe_stack_forward(stack, ctypes.byref(_input(x, token_ids)), _p(out), _p(scratch),
                                                     _stream(stream)))


def moe_stack_destroy(stack) -> None:
    if stack:
        lib().moe_stack_destroy(stack)


def moe_mx_blocks_unpack(blocks: torch.Tensor, nibble_order: int, stream=None):
    """17-byte MXFP4 blocks (uint8, 17 * n bytes) -> (codes uint8 [n, 16], scales uint8 [n])."""
    n = blocks.numel() // 17
    codes = torch.empty((n, 16), dtype=torch.uint8, device=blocks.device)
    scales = torch.empty((n,), dtype=torch.uint8, device=blocks.device)
    _ok("moe_mx_blocks_unpack", lib().moe_mx_blocks_unpack(_p(blocks), n, int(nibble_order), _p(codes), _p(scales),
                                                           _stream(stream)))
    return codes, scales


def moe_experts_destroy(h) -> None:
    if h:
        lib().moe_experts_destroy(h)


class _DeviceView:
    """__cuda_array_interface__ over library-owned device memory (read through torch.as_tensor)."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape), "typestr": typestr,
                                         "version": 3, "strides": None}
        self._owner = owner


# ----------------------------------------------------------------------------- convenience layer
@dataclass
class DeviceExperts:
    w13: torch.Tensor   # uint8 [n, 2f, d/2]
    s13: torch.Tensor   # uint8 [n, 2f, d/32]
    w2: torch.Tensor    # uint8 [n, d, f/2]
    s2: torch.Tensor    # uint8 [n, d, f/32]


def _to_dev(a, device) -> torch.Tensor:
    return torch.from_numpy(a).to(device) if not isinstance(a, torch.Tensor) else a.to(device)


class MoELayer:
    """One MoE layer resident on a GPU: routed and shared expert handles, router (or hash table),
    and a workspace sized for ``max_T`` rows.  ``forward`` is one ``moe_forward`` call."""

    def __init__(self, d_model, d_ff, n_experts, top_k, experts: DeviceExperts, shared: DeviceExperts | None,
                 router_w: torch.Tensor | None, router_bias: torch.Tensor | None,
                 hash_table: torch.Tensor | None = None, max_T: int = 512, route_scale: float = 1.5,
                 swiglu_limit: float = 10.0, device=None, act: str = "mxfp8", resident_router: bool = False):
        self.device = torch.device(device or "cuda")
        self.act = act
        self.resident_router = resident_router and router_w is not None
        self.cfg = make_config(d_model, d_ff, n_experts, top_k, route_scale, swiglu_limit)
        self.d, self.f, self.E, self.k, self.max_T = d_model, d_ff, n_experts, top_k, max_T
        self.experts, self.shared_w = experts, shared
        self.router_w, self.router_bias, self.hash_table = router_w, router_bias, hash_table
        self._handles = []
        with torch.cuda.device(self.device):
            self.h = moe_experts_create(self.cfg, n_experts, experts.w13, experts.s13, experts.w2, experts.s2)
            self._handles.append(self.h)
            self.h_shared = None
            if shared is not None:
                self.h_shared = moe_experts_create(self.cfg, 1, shared.w13, shared.s13, shared.w2, shared.s2)
                self._handles.append(self.h_shared)
            if hash_table is not None:
                moe_experts_set_hash_table(self.h, hash_table)
            for h in self._handles:
                moe_experts_set_activation_format(h, act)
            if self.resident_router:  # split once here; forward passes no router weights
                moe_experts_set_router(self.h, router_w, router_bias)
            nbytes = moe_workspace_size(self.cfg, max_T)
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            moe_set_workspace(self.h, self.workspace, max_T)
            torch.cuda.current_stream(self.device).synchronize()

    @classmethod
    def from_host(cls, inp, device=None, max_T: int | None = None, with_shared: bool = True,
                  act: str = "mxfp8", resident_router: bool = False) -> "MoELayer":
        """Build from host arrays (an object with the fields of ``synth.LayerInputs``); act is the
        activation format ("mxfp8", or "mxfp4" for the MXFP4-activation variant)."""
        dev = torch.device(device or "cuda")
        wl = inp.wl
        ex = DeviceExperts(*(_to_dev(getattr(inp.experts, n), dev) for n in ("w13", "s13", "w2", "s2")))
        sh = None
        if with_shared and inp.shared is not None:
            sh = DeviceExperts(*(_to_dev(getattr(inp.shared, n), dev) for n in ("w13", "s13", "w2", "s2")))
        rw = None if inp.router_w is None else _to_dev(inp.router_w, dev)
        rb = None if inp.router_bias is None else _to_dev(inp.router_bias, dev)
        tab = None if inp.hash_table is None else _to_dev(inp.hash_table, dev)
        layer = cls(wl.d, wl.f, wl.E, wl.k, ex, sh, rw, rb, tab, max_T or wl.T, wl.route_scale, wl.swiglu_limit, dev,
                    act, resident_router)
        layer.token_ids = None if inp.token_ids is None else _to_dev(inp.token_ids, dev)
        return layer

    def forward(self, x: torch.Tensor, token_ids: torch.Tensor | None = None, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
        if token_ids is None and self.hash_table is not None:
            token_ids = self.token_ids
        if out is None:
            out = torch.empty((x.shape[0], self.d), dtype=torch.bfloat16, device=self.device)
        rw, rb = (None, None) if self.resident_router else (self.router_w, self.router_bias)
        moe_forward(x, rw, rb, self.h, self.h_shared, out, token_ids, stream)
        return out

    def route(self, x: torch.Tensor, token_ids: torch.Tensor | None = None):
        if token_ids is None and self.hash_table is not None:
            token_ids = self.token_ids
        T = x.shape[0]
        ids = torch.empty((T, self.k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=self.device)
        rw, rb = (None, None) if self.resident_router else (self.router_w, self.router_bias)
        moe_route(self.h, x, rw, rb, ids, w, token_ids)
        return ids, w

    def permute(self, x: torch.Tensor, ids: torch.Tensor):
        T = x.shape[0]
        R = T * self.k
        dev = self.device
        out = dict(counts=torch.empty(self.E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                   perm_tok=torch.empty(R, dtype=torch.int32, device=dev),
                   inv_pos=torch.empty((T, self.k), dtype=torch.int32, device=dev),
                   a_q=torch.empty((R, self.d // 2 if self.act == "mxfp4" else self.d), dtype=torch.uint8,
                                   device=dev),
                   a_s=torch.empty((R, self.d // 32), dtype=torch.uint8, device=dev))
        moe_permute(self.h, x, ids, out["counts"], out["offsets"], out["perm_tok"], out["inv_pos"], out["a_q"],
                    out["a_s"])
        return out

    def expert_ffn(self, a_q, a_s, offsets=None, row_w=None, shared: bool = False) -> torch.Tensor:
        h = self.h
        if shared:
            h = self.h_shared
            if getattr(self, "_shared_ws", None) is None:  # the shared handle gets a workspace on first use
                self._shared_ws = torch.empty(moe_workspace_size(self.cfg, self.max_T), dtype=torch.uint8,
                                              device=self.device)
                moe_set_workspace(h, self._shared_ws, self.max_T)
        y = torch.empty((a_q.shape[0], self.d), dtype=torch.bfloat16, device=self.device)
        moe_expert_ffn(h, int(a_q.shape[0]), offsets, a_q, a_s, row_w, y)
        return y

    def last_routing(self):
        ids_p, w_p, T = moe_get_routing(self.h)
        ids = torch.as_tensor(_DeviceView(ids_p, (T, self.k), "<i4", self), device=self.device)
        w = torch.as_tensor(_DeviceView(w_p, (T, self.k), "<f4", self), device=self.device)
        return ids.clone(), w.clone()

    def last_h(self, shared: bool = False):
        """(codes, scales) of h from the last forward / expert_ffn (test hook)."""
        with torch.cuda.device(self.device):
            return moe_testing_read_h(self.h_shared if shared else self.h, self.f, self.act)

    def last_y32(self) -> torch.Tensor:
        """The last forward's output before its rounding to bf16, fp32 [T, d] (test hook)."""
        with torch.cuda.device(self.device):
            return moe_testing_read_y32(self.h, self.d)

    def last_topk_ids(self) -> torch.Tensor:
        return self.last_routing()[0]

    def check(self) -> None:
        moe_check(self.h)
        if self.h_shared is not None:
            moe_check(self.h_shared)

    def close(self) -> None:
        for h in self._handles:
            moe_experts_destroy(h)
        self._handles = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoEStack:
    """Layers run back to back by ``moe_stack_forward``: x_{l+1} = bf16(x_l + layer_l(x_l)).

    ``layers`` are ``MoELayer`` objects (they keep their own handles and weights); all of them get one
    shared workspace for ``max_T`` rows (or one each with ``separate_workspaces``, which keeps every
    layer's routing readable after a forward), and the stack owns the scratch buffer of the residual
    stream.  With ``use_graph`` the whole stack is captured once into a CUDA graph and replayed."""

    def __init__(self, layers, max_T: int, use_graph: bool = True, device=None, separate_workspaces: bool = False):
        self.layers = list(layers)
        self.device = torch.device(device or self.layers[0].device)
        self.d, self.max_T = self.layers[0].d, max_T
        with torch.cuda.device(self.device):
            nbytes = max(moe_workspace_size(ly.cfg, max_T) for ly in self.layers)
            n_ws = len(self.layers) if separate_workspaces else 1
            self.workspaces = [torch.empty(nbytes, dtype=torch.uint8, device=self.device) for _ in range(n_ws)]
            for i, ly in enumerate(self.layers):
                moe_set_workspace(ly.h, self.workspaces[i % n_ws], max_T)
            self.scratch = torch.empty((max_T, self.d), dtype=torch.bfloat16, device=self.device)
            self.stack = moe_stack_create([(ly.h, ly.h_shared, *((None, None) if ly.resident_router else
                                                                 (ly.router_w, ly.router_bias)))
                                           for ly in self.layers],
                                          use_graph)

    def forward(self, x: torch.Tensor, token_ids: torch.Tensor | None = None, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((x.shape[0], self.d), dtype=torch.bfloat16, device=self.device)
        moe_stack_forward(self.stack, x, out, self.scratch[: x.shape[0]], token_ids, stream)
        return out

    def check(self) -> None:
        for ly in self.layers:
            ly.check()

    def close(self) -> None:
        if getattr(self, "stack", None):
            moe_stack_destroy(self.stack)
            self.stack = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
