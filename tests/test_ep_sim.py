"""Expert-parallel dispatch / combine plan (block_scaled_fp4_sqrt_gb300.ep), simulated with CPU ranks.

Two gloo ranks each hold half of the tokens and half of the routed experts.  Rows travel to the owner
of their expert with all_to_all, the owner runs the oracle's grouped FFN on its experts in the plan's
order, the rows travel back, and the source sums them in the fixed slot order plus the shared row.
The result must equal the single-process oracle layer.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WL = dict(T=32, d=256, f=128, E=8, k=2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer_inputs():
    import oracle
    import synth
    wl = synth.Workload("ep_sim", WL["T"], WL["d"], WL["f"], WL["E"], WL["k"])
    inp = synth.gen_layer(wl, 21)
    ids, wts, _ = oracle.route(inp.x, inp.router_w, inp.router_bias, wl.k, wl.route_scale)
    return wl, inp, ids, wts


def _a2a(send: torch.Tensor, send_counts, recv_counts) -> torch.Tensor:
    import torch.distributed as dist
    recv = torch.empty((int(sum(recv_counts)),) + tuple(send.shape[1:]), dtype=send.dtype)
    dist.all_to_all_single(recv, send.contiguous(), [int(c) for c in recv_counts], [int(c) for c in send_counts])
    return recv


def _ep_rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import oracle
    import synth
    from block_scaled_fp4_sqrt_gb300 import ep
    wl, inp, ids, wts = _layer_inputs()
    T_r = wl.T // world
    tok = slice(rank * T_r, (rank + 1) * T_r)
    q, s = oracle.quantize_x(inp.x[tok])
    my_ids, my_w = ids[tok], wts[tok]
    plan = ep.plan_dispatch(my_ids, wl.E, world)
    src_tok = plan.order // wl.k
    # dispatch: the sizes first, then rows, scales, weights and expert ids
    recv_counts = _a2a(torch.from_numpy(plan.counts), [1] * world, [1] * world).numpy()
    rq = _a2a(torch.from_numpy(q[src_tok]), plan.counts, recv_counts).numpy()
    rs = _a2a(torch.from_numpy(s[src_tok]), plan.counts, recv_counts).numpy()
    rw = _a2a(torch.from_numpy(my_w.reshape(-1)[plan.order].astype(np.float64)), plan.counts, recv_counts).numpy()
    re = _a2a(torch.from_numpy(plan.expert), plan.counts, recv_counts).numpy()
    # the owner's grouped FFN over its own experts, in the plan's expert-major order
    rp = ep.plan_receive(re, recv_counts, wl.E, world, rank)
    per = wl.E // world
    lo = rank * per
    mine = synth.ExpertWeights(*(getattr(inp.experts, n)[lo:lo + per] for n in ("w13", "s13", "w2", "s2")))
    y_c, _, _ = oracle.expert_ffn(rq[rp.order], rs[rp.order], mine, offsets=rp.offsets, row_w=rw[rp.order])
    y_arrival = np.empty_like(y_c)
    y_arrival[rp.order] = y_c
    # combine: rows back to their source, summed in slot order plus the shared row
    back = _a2a(torch.from_numpy(y_arrival), recv_counts, plan.counts).numpy()
    sh, _, _ = oracle.expert_ffn(q, s, inp.shared)
    y = ep.combine_rows(back, plan, T_r, wl.k, sh)
    np.save(os.path.join(out_dir, f"y{rank}.npy"), y)
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def built():
    import __graft_entry__ as g
    g.build_cpu()


def test_plan_orders_rows_by_destination_expert_token():
    sys.path.insert(0, ROOT)
    from block_scaled_fp4_sqrt_gb300 import ep
    ids = np.array([[5, 1], [0, 6], [1, 4]])
    plan = ep.plan_dispatch(ids, 8, 2)
    # rank 0 owns experts 0..3: (t1, e0), (t0, e1), (t2, e1); rank 1: (t2, e4), (t0, e5), (t1, e6)
    assert plan.counts.tolist() == [3, 3]
    assert plan.order.tolist() == [2, 1, 4, 5, 0, 3]
    assert plan.expert.tolist() == [0, 1, 1, 4, 5, 6]
    rp = ep.plan_receive(np.array([4, 5, 6, 5]), np.array([3, 1]), 8, 2, 1)
    assert rp.order.tolist() == [0, 1, 3, 2] and rp.offsets.tolist() == [0, 1, 3, 4, 4]
    with pytest.raises(ValueError):
        ep.plan_receive(np.array([1]), np.array([1]), 8, 2, 1)


def test_two_rank_expert_parallel_layer_equals_the_oracle(built, tmp_path):
    import oracle
    port = _free_port()
    mp.start_processes(_ep_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    y = np.concatenate([np.load(tmp_path / "y0.npy"), np.load(tmp_path / "y1.npy")])
    wl, inp, ids, wts = _layer_inputs()
    y_ref = oracle.layer(inp.x, ids, wts, inp.experts, inp.shared, wl.swiglu_limit)
    scale = np.abs(y_ref).max()
    assert np.max(np.abs(y - y_ref)) <= 1e-12 * scale
