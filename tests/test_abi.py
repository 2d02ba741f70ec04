"""The C-ABI library builds, loads and exports every symbol its headers declare; host-side argument
checks answer without a GPU (no compute call is made here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libmoe():
    import __graft_entry__ as g
    g.build_cuda()
    import block_scaled_fp4_sqrt_gb300 as m
    return m


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names.update(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\(", open(h).read(), flags=re.M))
    return names


def test_headers_declare_the_layer_calls():
    names = _declared()
    for must in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_forward"):
        assert must in names


def test_every_declared_symbol_is_exported(libmoe):
    L = libmoe.lib()
    missing = [n for n in sorted(_declared()) if not hasattr(L, n)]
    assert not missing, missing
    assert set(libmoe.EXPORTED) == _declared()


def test_host_side_validation_without_gpu(libmoe):
    L = libmoe.lib()
    cfg = libmoe.make_config(4096, 2048, 256, 6)
    h = ctypes.c_void_p()
    assert L.moe_experts_create(ctypes.byref(cfg), 0, None, None, None, None, None, ctypes.byref(h)) == 1
    assert b"expert count" in L.moe_last_error()
    assert L.moe_experts_create(ctypes.byref(cfg), 256, None, None, None, None, None, ctypes.byref(h)) == 1
    misaligned = ctypes.c_void_p(4096 + 8)
    ok_ptr = ctypes.c_void_p(4096)
    assert L.moe_experts_create(ctypes.byref(cfg), 256, misaligned, ok_ptr, ok_ptr, ok_ptr, None, ctypes.byref(h)) == 1
    assert b"16-byte" in L.moe_last_error()
    for bad in (libmoe.make_config(4000, 2048, 256, 6), libmoe.make_config(4096 + 128, 2048, 256, 6),
                libmoe.make_config(4096, 2048, 256, 17),
                libmoe.make_config(4096, 2048, 4, 6), libmoe.make_config(4096, 100, 256, 6)):
        assert L.moe_experts_create(ctypes.byref(bad), 1, ok_ptr, ok_ptr, ok_ptr, ok_ptr, None, ctypes.byref(h)) == 2
        assert libmoe.moe_workspace_size(bad, 512) == 0
    assert L.moe_forward(None, None, None, None, None, None, None) == 1
    assert L.moe_check(None, None) == 1
    assert L.moe_set_workspace(None, None, 0, 1) == 1
    assert L.moe_status_string(6) == b"device wait timed out"
    st = ctypes.c_void_p()
    assert L.moe_stack_create(None, 0, 0, ctypes.byref(st)) == 1 and not st.value
    assert L.moe_stack_forward(None, None, None, None, None) == 1
    assert L.moe_experts_set_activation_format(None, libmoe.MOE_ACT_MXFP4) == 1
    assert L.moe_experts_set_router(None, None, None, None) == 1
    n = ctypes.c_int32(-1)
    assert L.moe_testing_read_h(None, None, None, ctypes.byref(n), None) == 1


def test_workspace_size_grows_with_T(libmoe):
    cfg = libmoe.make_config(4096, 2048, 256, 6)
    sizes = [libmoe.moe_workspace_size(cfg, T) for T in (1, 8, 512, 8192)]
    assert all(a < b for a, b in zip(sizes, sizes[1:]))
    # the dominant terms: activations, h and the bf16 expert rows, (k + 1) rows per token
    assert sizes[-1] >= 8192 * 7 * (4096 + 2048 + 2 * 4096)
