"""The expert-parallel plan (block_scaled_fp4_sqrt_gb300.ep) on the CUDA path: two gloo ranks on one GPU,
each holding half of the tokens and a handle with half of the routed experts.

* Source side: moe_permute quantises the rank's tokens to MXFP8 and orders the (token, slot) rows
  expert-major with tokens ascending.  Because expert ownership is a contiguous block per rank, that is
  exactly the plan's send order (destination, expert, token, slot), which the test checks row by row.
* The rows, their scales, routing weights and expert ids travel to their owners with all_to_all on the
  host (gloo); the owner runs moe_expert_ffn over its own experts in the plan's receive order and
  returns the bf16 rows in arrival order.
* The source sums each token's slots in order 0..k-1 plus its shared-expert row (moe_expert_ffn on the
  shared handle), in fp64, and the result is compared with the single-process fp64 oracle layer.

The rows cross the ranks in bf16, so the bound is the layer's (2e-2 rms) plus each summed row's own
rounding (2^-8 of its magnitude).  Nothing here waits on another rank on the device: the ranks exchange
data only through the host.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

WL = dict(T=128, d=512, f=256, E=16, k=4)
WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer_inputs():
    import oracle
    import synth
    wl = synth.Workload("ep_gpu", WL["T"], WL["d"], WL["f"], WL["E"], WL["k"])
    inp, ids, wts, _ = oracle.margin_filtered_layer(wl, seed=23)
    return wl, inp, ids, wts


def _a2a(send: np.ndarray, send_counts, recv_counts) -> np.ndarray:
    import torch.distributed as dist
    s = torch.from_numpy(np.ascontiguousarray(send))
    recv = torch.empty((int(sum(recv_counts)),) + tuple(s.shape[1:]), dtype=s.dtype)
    dist.all_to_all_single(recv, s, [int(c) for c in recv_counts], [int(c) for c in send_counts])
    return recv.numpy()


def _ep_gpu_rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import block_scaled_fp4_sqrt_gb300 as m
    from block_scaled_fp4_sqrt_gb300 import ep
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl, inp, ids, wts = _layer_inputs()
    T_r, k, E, d = wl.T // world, wl.k, wl.E, wl.d
    per = E // world
    lo = rank * per

    def to(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    cfg = m.make_config(d, wl.f, E, k)
    h = m.moe_experts_create(cfg, per, *(to(getattr(inp.experts, n)[lo:lo + per]) for n in ("w13", "s13", "w2", "s2")))
    hs = m.moe_experts_create(cfg, 1, *(to(getattr(inp.shared, n)) for n in ("w13", "s13", "w2", "s2")))
    try:
        wss = [torch.empty(m.moe_workspace_size(cfg, wl.T), dtype=torch.uint8, device=dev) for _ in range(2)]
        m.moe_set_workspace(h, wss[0], wl.T)
        m.moe_set_workspace(hs, wss[1], wl.T)
        # source side: MXFP8 rows of this rank's tokens in expert-major order, on the GPU
        tok = slice(rank * T_r, (rank + 1) * T_r)
        my_ids, my_w = ids[tok], wts[tok]
        R = T_r * k
        x = to(inp.x[tok].view(np.int16)).view(torch.bfloat16)
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(R, dtype=torch.int32, device=dev)
        inv = torch.empty((T_r, k), dtype=torch.int32, device=dev)
        a_q = torch.empty((R, d), dtype=torch.uint8, device=dev)
        a_s = torch.empty((R, d // 32), dtype=torch.uint8, device=dev)
        m.moe_permute(h, x, to(my_ids), counts, offsets, perm, inv, a_q, a_s)
        torch.cuda.synchronize()
        m.moe_check(h)
        plan = ep.plan_dispatch(my_ids, E, world)
        inv_np = inv.cpu().numpy()
        flat_of_row = np.empty(R, dtype=np.int64)
        flat_of_row[inv_np.reshape(-1)] = np.arange(R)
        assert np.array_equal(flat_of_row, plan.order), "the GPU permutation is not the plan's send order"
        # dispatch through the host
        recv_counts = _a2a(plan.counts, [1] * world, [1] * world)
        rq = _a2a(a_q.cpu().numpy(), plan.counts, recv_counts)
        rs = _a2a(a_s.cpu().numpy(), plan.counts, recv_counts)
        rw = _a2a(my_w.reshape(-1)[plan.order].astype(np.float32), plan.counts, recv_counts)
        re = _a2a(plan.expert, plan.counts, recv_counts)
        # the owner's grouped FFN over its experts, in the plan's expert-major order
        rp = ep.plan_receive(re, recv_counts, E, world, rank)
        n = rq.shape[0]
        y = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
        m.moe_expert_ffn(h, n, to(rp.offsets.astype(np.int32)), to(rq[rp.order]), to(rs[rp.order]),
                         to(rw[rp.order]), y)
        torch.cuda.synchronize()
        m.moe_check(h)
        y_arrival = np.empty((n, d), dtype=np.float32)
        y_arrival[rp.order] = y.float().cpu().numpy()
        back = _a2a(y_arrival, recv_counts, plan.counts).astype(np.float64)
        # the shared expert on this rank's own tokens: slot 0's rows are the tokens' MXFP8 rows
        rows0 = torch.from_numpy(inv_np[:, 0].astype(np.int64)).to(dev)
        ysh = torch.empty((T_r, d), dtype=torch.bfloat16, device=dev)
        m.moe_expert_ffn(hs, T_r, None, a_q[rows0].contiguous(), a_s[rows0].contiguous(), None, ysh)
        torch.cuda.synchronize()
        m.moe_check(hs)
        ysh_np = ysh.float().cpu().numpy().astype(np.float64)
        out = ep.combine_rows(back, plan, T_r, k, ysh_np)
        absum = ep.combine_rows(np.abs(back), plan, T_r, k, np.abs(ysh_np))
        np.save(os.path.join(out_dir, f"y{rank}.npy"), out)
        np.save(os.path.join(out_dir, f"a{rank}.npy"), absum)
    finally:
        m.moe_experts_destroy(h)
        m.moe_experts_destroy(hs)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_expert_parallel_layer_on_the_gpu(tmp_path):
    import __graft_entry__ as g
    g.build()
    import oracle
    from gpu_support import TOL_MAX_RMS, TOL_MEAN_REL
    port = _free_port()
    mp.start_processes(_ep_gpu_rank, args=(WORLD, port, str(tmp_path)), nprocs=WORLD, join=True,
                       start_method="spawn")
    y = np.concatenate([np.load(tmp_path / f"y{r}.npy") for r in range(WORLD)])
    absum = np.concatenate([np.load(tmp_path / f"a{r}.npy") for r in range(WORLD)])
    wl, inp, ids, wts = _layer_inputs()
    y_ref = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, wl.swiglu_limit)
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = np.abs(y - y_ref)
    rounding = 2.0 ** -8 * absum
    print(f"EP on the GPU: max |dy| / rms = {err.max() / rms:.3e}, mean rel = {err.sum() / np.abs(y_ref).sum():.3e}")
    assert np.all(err <= TOL_MAX_RMS * rms + rounding)
    assert err.sum() <= TOL_MEAN_REL * np.abs(y_ref).sum() + rounding.sum()
