"""moe_route_noalloc: the learned router for callers that can't call cudaMalloc (under a host framework
that owns all device memory, on paths that must not enter an allocator).  It keeps its scratch in a
fixed array of library device memory instead of a workspace.

Checked here through the C ABI against moe_route (the handle + workspace entry point) and against the
oracle's routing on two calls in a row with different batch sizes, so the second call runs over the
scratch the first one left; and the size limit of the fixed scratch.  This file runs last so that a failure here, under `-x`, stops
only after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_WEIGHT_REL = 1e-4  # the routing-weight tolerance of the parity tests


def _router_inputs(seed, T, d, E, k):
    """x rows redrawn until no top-k selection gap is below the oracle's margin: moe_route and
    moe_route_noalloc add their fp32 products in different orders, and only the order of exact
    near-ties could otherwise separate their expert ids."""
    rw, rb, _ = synth.gen_router(seed, E, d)
    x = synth.gen_x(seed, T, d)
    attempts = np.zeros(T, np.int32)
    for _ in range(64):
        ids, wts, margin = oracle.route(x, rw, rb, k)
        low = np.nonzero(margin < oracle.MARGIN_MIN)[0]
        if low.size == 0:
            break
        attempts[low] += 1
        x[low] = synth.gen_x(seed, T, d, attempts)[low]
    else:
        raise RuntimeError("margin rejection did not converge")
    return x, rw, rb, ids, wts


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__ as g
    g.build_cuda()
    import block_scaled_fp4_sqrt_gb300 as m
    return m


def test_noalloc_router_matches_moe_route_on_two_calls_in_a_row(moe):
    dev = torch.device("cuda:0")
    d, f, E, k, max_T = 4096, 128, 256, 6, 512
    cfg = moe.make_config(d, f, E, k)
    # the handle moe_route needs; expert weight contents do not enter the routing
    w13 = torch.zeros((E, 2 * f, d // 2), dtype=torch.uint8, device=dev)
    s13 = torch.full((E, 2 * f, d // 32), 127, dtype=torch.uint8, device=dev)
    w2 = torch.zeros((E, d, f // 2), dtype=torch.uint8, device=dev)
    s2 = torch.full((E, d, f // 32), 127, dtype=torch.uint8, device=dev)
    h = moe.moe_experts_create(cfg, E, w13, s13, w2, s2)
    try:
        ws = torch.empty(moe.moe_workspace_size(cfg, max_T), dtype=torch.uint8, device=dev)
        moe.moe_set_workspace(h, ws, max_T)
        for seed, T in ((11, 512), (12, 300)):
            xb, rw, rb, ids_orc, wts_orc = _router_inputs(seed, T, d, E, k)
            router_w = torch.from_numpy(rw).to(dev)
            router_b = torch.from_numpy(rb).to(dev)
            x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
            ids_ref = torch.empty((T, k), dtype=torch.int32, device=dev)
            w_ref = torch.empty((T, k), dtype=torch.float32, device=dev)
            moe.moe_route(h, x, router_w, router_b, ids_ref, w_ref)
            ids = torch.full((T, k), -1, dtype=torch.int32, device=dev)
            w = torch.full((T, k), -1.0, dtype=torch.float32, device=dev)
            moe.moe_route_noalloc(cfg, x, router_w, router_b, ids, w)
            torch.cuda.synchronize()
            assert torch.equal(ids, ids_ref), f"T={T}: expert ids differ"
            rel = ((w - w_ref).abs() / w_ref.abs()).max().item()
            assert rel <= TOL_WEIGHT_REL, f"T={T}: routing weights differ by {rel:.3e}"
            # and against the fp64 oracle directly: ids bit for bit, weights within the same bound
            assert np.array_equal(ids.cpu().numpy(), ids_orc), f"T={T}: expert ids differ from the oracle's"
            w_np = w.cpu().numpy().astype(np.float64)
            rel_o = np.max(np.abs(w_np - wts_orc) / np.abs(wts_orc))
            assert rel_o <= TOL_WEIGHT_REL, f"T={T}: routing weights differ from the oracle's by {rel_o:.3e}"
        moe.moe_check(h)
    finally:
        moe.moe_experts_destroy(h)


def test_noalloc_router_rejects_batches_beyond_its_scratch(moe):
    dev = torch.device("cuda:0")
    d, E, k = 4096, 256, 6
    cfg = moe.make_config(d, 128, E, k)
    T = 4097  # T * E = 1,048,832 > 1,048,576 scratch values
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    rw = torch.zeros((E, d), dtype=torch.float32, device=dev)
    rb = torch.zeros((E,), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    with pytest.raises(moe.MoEError) as err:
        moe.moe_route_noalloc(cfg, x, rw, rb, ids, w)
    assert err.value.status == 3 and "exceeds the fixed scratch" in str(err.value)
