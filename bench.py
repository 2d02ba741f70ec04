#!/usr/bin/env python3
"""Benchmark of the MoE-layer forward on GB300: tokens/s at a verify batch, with the roofline of the
dominant kernel, an end-to-end leg through host buffers, and the fp64 oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload verify512] [--impl ours|reference]

One step = one moe_forward (route -> dispatch -> gate-up GEMM -> down GEMM -> combine) over one batch of
synthetic token rows; the expert weights (3.44 GB for verify512) are resident in HBM and larger than L2,
so no flush is needed between steps.  Under torchrun every rank runs its own replica on its own batch
(weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/sec at T=512 verify; achieved HBM GB/s / tensor-pipe %"


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="verify512")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--act", choices=["mxfp8", "mxfp4"], default="mxfp8",
                   help="activation format: the layer's MXFP8, or the MXFP4-activation variant (kind::mxf4)")
    p.add_argument("--experts", type=int, default=0,
                   help="override the routed-expert count (small cases for profiling; not a benchmark line)")
    p.add_argument("--tokens", type=int, default=0, help="override T (small cases for profiling)")
    p.add_argument("--layers", type=int, default=1,
                   help="> 1: time a stack of this many MoE layers (moe_stack_forward) instead of one layer")
    p.add_argument("--hash-layers", type=int, default=3, help="hash-routed layers at the bottom of the stack")
    p.add_argument("--workloads", default="all",
                   help="after the headline, also measure these workloads into the line's 'workloads' object: "
                        "'all' (the five layer configurations), 'none', or a comma-separated list (one GPU only)")
    p.add_argument("--pair-gemm", action="store_true",
                   help="run 128-row tiles on the CTA-pair grouped GEMMs instead of the one-SM kernels (A/B comparisons)")
    p.add_argument("--cpu-seconds-other", type=float, default=4.0,
                   help="target CPU time of the oracle baseline sample of each extra workload")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def replica_x(seed: int, rank: int, world: int, T: int, d: int):
    """Each replica's own batch of token rows: with one GPU the workload's batch, under torchrun rank r
    draws from seed + 7919 r (rank 0 keeps the one-GPU batch)."""
    import synth
    return synth.gen_x(seed + 7919 * rank if world > 1 else seed, T, d)


def init_replicas(backend: str, timeout_s: float = 300.0) -> None:
    """Join the torchrun job (RANK / WORLD_SIZE / MASTER_ADDR / MASTER_PORT from the environment).  A
    finite timeout makes a barrier or reduction whose peer has died end in an error, not a hang."""
    import datetime

    import torch.distributed as dist
    dist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (all-reduce MAX of one scalar); x itself on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, T: int, ms_per_step: float) -> float:
    """Whole-job throughput: every replica processes T tokens per step; the slowest rank's time counts."""
    return world * T / (ms_per_step * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            m = json.load(fh)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def expert_bytes(wl):
    """MXFP4 bytes of one expert: gate + up + down codes (0.5 B each) plus one E8M0 byte per 32."""
    n = 3 * wl.d * wl.f
    return n // 2 + n // 32


def stage_bytes(wl, touched, rows, act: str = "mxfp8"):
    """Algorithmic HBM bytes per launch of each stage (touched = experts read, including the shared one).
    Activation rows (A, H) take one byte per element in MXFP8 and half a byte in MXFP4; the weighted expert
    rows between the down GEMM and the combine take two bytes per element plus a scale byte per 32."""
    d, f, T, k, E = wl.d, wl.f, wl.T, wl.k, wl.E
    per = 2 if act == "mxfp4" else 1
    gate_up_w = 2 * f * d // 2 + 2 * f * d // 32
    down_w = d * f // 2 + d * f // 32
    router = (0 if wl.hashed else E * d * 4 + E * 4) + T * d * 2 + T * k * 8
    return {
        "route": router,
        "dispatch": T * d * 2 + rows * (d // per + d // 32),
        "gemm_gate_up": touched * gate_up_w + rows * (d // per + d // 32) + rows * (f // per + f // 32),
        "gemm_down": touched * down_w + rows * (f // per + f // 32) + rows * (2 * d + d // 32),
        "combine": rows * (2 * d + d // 32) + T * d * 2,
    }


def layer_bytes(wl, touched):
    b = touched * expert_bytes(wl) + 2 * wl.T * wl.d * 2
    if wl.hashed:
        b += wl.T * 4 + wl.T * wl.k * 4
    else:
        b += wl.E * wl.d * 4 + wl.E * 4
    return b


def gemm_flops(wl, rows):
    return {"gemm_gate_up": 2 * rows * 2 * wl.f * wl.d, "gemm_down": 2 * rows * wl.d * wl.f}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# sources that decide what the grouped GEMMs read and write (kernel, launch shape, work list, weight layout)
GEMM_SOURCES = ("moe_gemm.cu", "moe_device.cuh", "moe_internal.h", "moe_api.cu", "moe_dispatch.cu", "moe_pack.cu")


def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp4_sqrt_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed ncu
    summary profiles/dram_traffic.txt, only if the GEMM sources have not changed since the capture.
    Lines: "digest <hex>" and "<workload> <kernel> <bytes> <note...>"."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest, table = None, {}
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "digest" and len(parts) > 1:
                digest = parts[1]
            elif len(parts) >= 3:
                table[(parts[0], parts[1])] = int(parts[2])
    if digest != kernel_source_digest():
        return None
    return table.get((workload, kernel))


def oracle_tokens_per_s(inp, wl, n_tokens: int, seed: int, act: str = "mxfp8"):
    """Time the fp64 oracle (routing + layer) on n_tokens sampled token rows."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(wl.T, size=min(n_tokens, wl.T), replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    if wl.hashed:
        ids, wts = oracle.hash_route(inp.token_ids[toks], inp.hash_table, wl.k, wl.route_scale)
    else:
        ids, wts, _ = oracle.route(inp.x[toks], inp.router_w, inp.router_bias, wl.k, wl.route_scale)
    oracle.layer(inp.x[toks], ids, wts, inp.experts, inp.shared, wl.swiglu_limit, act=act)
    dt = time.perf_counter() - t0
    return len(toks), dt


def cpu_baseline(inp, wl, target_s: float, seed: int, act: str = "mxfp8"):
    import oracle
    n0 = 4
    _, t0 = oracle_tokens_per_s(inp, wl, n0, seed, act)
    n = int(max(n0, min(wl.T, round(target_s / max(t0 / n0, 1e-9)))))
    n, dt = oracle_tokens_per_s(inp, wl, n, seed + 1, act)
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{n} of the {wl.T} token rows of {wl.name} (routing + all expert rows + combine), fp64, {dt:.1f} s"}


def run_reference(args, wl):
    """Reference arm: the fp64 oracle as it stands, on the host cores, same workload and metric."""
    import synth
    rank, _, world = dist_env()
    if rank != 0:
        return
    inp = synth.gen_layer(wl, args.seed)
    import oracle
    per_step = max(1, min(wl.T, 4 if wl.d >= 4096 else 16))
    for i in range(args.warmup):
        oracle_tokens_per_s(inp, wl, per_step, 1000 + i, args.act)
    total_tok, total_s = 0, 0.0
    for i in range(args.steps):
        n, dt = oracle_tokens_per_s(inp, wl, per_step, 2000 + i, args.act)
        total_tok += n
        total_s += dt
    value = total_tok / total_s
    cores = oracle.threads()
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(wl, args.act),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} token rows of {wl.name} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def layer_launches(wl) -> int:
    """Kernels one layer forward launches with the router resident on the handle.  Route: the hash-table
    kernel, or the fused cluster router (up to 256 experts; above that tensor-core logits + a top-k kernel).
    Dispatch: histogram, column scan, group scan, gather -- for learned routing of up to 32 rows the router's
    last CTA writes the dispatch state and only the gather remains.  The two grouped GEMMs, then the combine."""
    small = not wl.hashed and wl.T <= 32
    route = 1 if (wl.hashed or small or wl.E <= 256) else 2  # router weights resident: no per-call split
    dispatch = 1 if small else 4
    return route + dispatch + 2 + 1


def workload_config(wl, act: str = "mxfp8"):
    return {"act": act, "workload": wl.name, "T": wl.T, "d_model": wl.d, "d_ff": wl.f, "routed_experts": wl.E, "top_k": wl.k,
            "shared_experts": 1, "routing": "hash table" if wl.hashed else "sqrt-softplus",
            "weights": "MXFP4 (E2M1 + E8M0/32), resident in HBM",
            "l2": "no flush: expert weights read per step exceed the 129 MB L2"}


def measure_layer(args, wl, inp, dev, world, rank, mx_peak, mma_name, cpu_target_s, headline):
    """Time one layer workload: device-timed steps, a staged pass, end-to-end legs and (one GPU) the oracle
    on the host cores.  Returns the record of this workload (the keys of the benchmark's JSON line)."""
    import numpy as np
    import torch

    import block_scaled_fp4_sqrt_gb300 as moe

    fp4 = args.act == "mxfp4"
    # the router weights are made resident once, like the expert weights (moe_experts_set_router)
    layer = moe.MoELayer.from_host(inp, device=dev, max_T=wl.T, act=args.act, resident_router=True)
    if args.pair_gemm:
        for h in (layer.h, layer.h_shared):
            moe.moe_testing_set_pair_gemm(h, True)
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        layer.forward(x, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    layer.check()
    ids, _ = layer.last_routing()
    touched = int(torch.unique(ids).numel()) + 1  # + shared expert
    rows = wl.T * wl.k + wl.T

    # ---- device-timed steps: plain steps back to back on the launching stream
    cvd = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    clocks = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else local_rank)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_begin.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    layer.check()
    ms = max_over_ranks(t_begin.elapsed_time(t_end) / args.steps, dev)

    # ---- per-stage times: a second live pass of the same steps with CUDA events between the stages
    # (an event between two kernels serialises them, so this pass runs slightly slower than the first)
    n_ev = moe.MOE_N_STAGES + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for ev in events:  # create the events before the timed region
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    keep = []
    for i in range(args.steps):
        keep.append(moe.moe_set_stage_events(layer.h, events[i]))
        step()
    torch.cuda.synchronize()
    moe.moe_set_stage_events(layer.h, None)
    layer.check()
    # medians over the steps: one step held up on the host (the events time the GPU between launches)
    # must not decide which kernel is the dominant one
    stage_ms = {name: statistics.median(ev[i].elapsed_time(ev[i + 1]) for ev in events)
                for i, name in enumerate(moe.STAGE_NAMES)}
    ms_staged = max_over_ranks(statistics.median(ev[0].elapsed_time(ev[-1]) for ev in events), dev)

    # ---- end to end: pinned host x in, bf16 out back to the host, every step.  The headline runs the steps
    # as a serving loop would: two device buffers, the H2D copy of step i+1 and the D2H copy of step i-1 on
    # their own streams while step i computes (each step's copies are inside the timed region; events order
    # every buffer reuse).  The serial variant (copy in, forward, copy out on one stream) is kept alongside.
    x_host = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_hosts = [torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    tok_dev = layer.token_ids
    tok_host = None if tok_dev is None else tok_dev.cpu().pin_memory()
    x_devs = [torch.empty_like(x) for _ in range(2)]
    out_devs = [torch.empty_like(out) for _ in range(2)]
    tok_devs = None if tok_dev is None else [torch.empty_like(tok_dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def h2d(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(ev_fwd[b])  # step i-2 has finished reading x_devs[b]
        with torch.cuda.stream(s_in):
            x_devs[b].copy_(x_host, non_blocking=True)
            if tok_host is not None:
                tok_devs[b].copy_(tok_host, non_blocking=True)
        ev_in[b].record(s_in)

    def compute_and_d2h(i):
        b = i % 2
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # the D2H of step i-2 has read out_devs[b]
        layer.forward(x_devs[b], token_ids=None if tok_devs is None else tok_devs[b], out=out_devs[b], stream=stream)
        ev_fwd[b].record(stream)
        s_out.wait_event(ev_fwd[b])
        with torch.cuda.stream(s_out):
            out_hosts[b].copy_(out_devs[b], non_blocking=True)
        ev_out[b].record(s_out)

    def pipelined(n):
        h2d(0)
        if n > 1:
            h2d(1)
        for i in range(n):
            compute_and_d2h(i)
            if i + 2 < n:
                h2d(i + 2)
        for b in range(min(n, 2)):
            stream.wait_event(ev_out[b])

    def serial_step():
        x_devs[0].copy_(x_host, non_blocking=True)
        if tok_host is not None:
            tok_devs[0].copy_(tok_host, non_blocking=True)
        layer.forward(x_devs[0], token_ids=None if tok_devs is None else tok_devs[0], out=out_devs[0])
        out_hosts[0].copy_(out_devs[0], non_blocking=True)

    def timed_e2e(body):
        body(3)  # warm-up
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        body(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)

    ms_e2e = timed_e2e(pipelined)
    layer.check()
    # the last step's result reached the host and equals the device-timed path's output (same x)
    assert torch.equal(out_hosts[(args.steps - 1) % 2], out.cpu()), "pipelined end-to-end output differs"
    ms_e2e_serial = timed_e2e(lambda n: [serial_step() for _ in range(n)])
    layer.close()
    del x_devs, out_devs, x, out

    pk = peaks()
    dom = max(stage_ms, key=stage_ms.get)
    sb = stage_bytes(wl, touched, rows, args.act)
    traffic_key = wl.name + (":mxfp4" if fp4 else "")  # rows of profiles/dram_traffic.txt
    fl = gemm_flops(wl, rows)
    # verify shapes stream the expert weights (HBM bound); with >= 64 rows per expert (the prefill
    # chunk) the grouped GEMMs are dense block-scaled contractions (tensor bound)
    compute_bound = wl.T * wl.k / wl.E >= 64
    if compute_bound and dom in fl:
        achieved = fl[dom] / (stage_ms[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": mx_peak, "unit": "TFLOP/s", "frac": achieved / mx_peak,
                "traffic": measured_traffic(dom, traffic_key), "kernel": dom,
                "peak_source": "measured in this run: back-to-back " + mma_name,
                "nominal_alt_peak": {"value": (6 if fp4 else 2) * pk["bf16_tflops_sustained"],
                                     "source": f"{pk['source']} bf16 sustained x {6 if fp4 else 2} (nominal "
                                               f"{'FP4' if fp4 else 'FP8'}/BF16 ratio)"},
                "algorithmic_flops_per_launch": fl[dom]}
    else:
        achieved = sb[dom] / (stage_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": measured_traffic(dom, traffic_key), "kernel": dom,
                "peak_source": f"{pk['source']} HBM copy bandwidth", "algorithmic_bytes_per_launch": sb[dom]}
    lb = layer_bytes(wl, touched)
    layer_fl = fl["gemm_gate_up"] + fl["gemm_down"]
    if compute_bound:
        layer_roof = {"bound": "tensor", "algorithmic_flops": layer_fl, "achieved": layer_fl / (ms * 1e-3) / 1e12,
                      "peak": mx_peak, "unit": "TFLOP/s", "frac": layer_fl / (ms * 1e-3) / 1e12 / mx_peak,
                      "peak_source": "measured in this run: back-to-back " + mma_name,
                      "how": "expert GEMM FLOPs of the whole layer (2 x 3 x d x f per routed and shared row) over "
                             "the whole step's time"}
        if fp4:
            layer_roof["frac_of_3x_mxf8f6f4_peak"] = None  # filled in by the caller
    elif lb < 64 << 20:  # a few launches over kilobytes to megabytes: bound by launch latency, not by HBM
        layer_roof = {"bound": "latency", "algorithmic_bytes": lb, "achieved": lb / (ms * 1e-3) / 1e9,
                      "peak": None, "unit": "GB/s", "frac": None,
                      "how": f"{layer_launches(wl)} dependent kernel launches over {lb / 1e6:.2f} MB"}
    else:
        layer_roof = {"bound": "hbm", "algorithmic_bytes": lb, "achieved": lb / (ms * 1e-3) / 1e9,
                      "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": lb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    rec = {
        "ms_per_step": ms, "value": job_tokens_per_s(world, wl.T, ms), "unit": "tokens/s",
        "config": dict(workload_config(wl, args.act), touched_experts=touched, parallelism=f"replicas x{world}",
                       gemm="CTA pairs" if args.pair_gemm and wl.T * wl.k > 16 * wl.E and not fp4 else "one-SM"),
        "roofline": roof,
        "layer_roofline": layer_roof,
        "gemm_tensor": {"achieved": layer_fl / ((stage_ms["gemm_gate_up"] + stage_ms["gemm_down"]) * 1e-3) / 1e12,
                        "peak": mx_peak, "unit": "TFLOP/s",
                        "frac": layer_fl / ((stage_ms["gemm_gate_up"] + stage_ms["gemm_down"]) * 1e-3) / 1e12 / mx_peak},
        "stage_ms": stage_ms,
        "stage_timing": {"ms_per_step": ms_staged, "how": "second pass of the same steps with CUDA events "
                         "between the stages (events serialise the launches there); medians over the steps"},
        "e2e": {"value": job_tokens_per_s(world, wl.T, ms_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.T * wl.d * 2 + (wl.T * 4 if wl.hashed else 0),
                "d2h_bytes_per_step": wl.T * wl.d * 2, "ms_per_step": ms_e2e,
                "how": "pinned host x -> device -> moe_forward -> pinned host out, every step; copies of steps i+1 "
                       "and i-1 overlap step i on their own streams (two device buffers)",
                "serial": {"value": job_tokens_per_s(world, wl.T, ms_e2e_serial), "ms_per_step": ms_e2e_serial,
                           "how": "copy in, forward, copy out on one stream"}},
        "gpu_launches": layer_launches(wl) * args.steps,
        "clocks": clk,
    }
    if world == 1 and cpu_target_s > 0:
        rec["cpu_baseline"] = cpu_baseline(inp, wl, cpu_target_s, args.seed, args.act)
    return rec


# The five layer configurations the layer is specified on; the default run measures all of them after the
# headline (verify512), reusing one draw of the full-size expert weights.
ALL_WORKLOADS = ("verify512", "verify8", "hash512", "prefill8192", "tiny")


def run_ours(args, wl):
    import torch

    import __graft_entry__ as g
    import synth

    rank, local_rank, world = dist_env()
    g.build()
    import block_scaled_fp4_sqrt_gb300 as moe

    if world > 1:
        init_replicas("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    inp = synth.gen_layer(wl, args.seed)
    if world > 1:  # each replica gets its own batch of token rows
        inp.x = replica_x(args.seed, rank, world, wl.T, wl.d)

    # block-scaled MMA peak of this GPU (the tensor roofline's denominator), before the timed region
    fp4 = args.act == "mxfp4"
    mx_peak = moe.moe_measure_mxf4_peak(4096) if fp4 else moe.moe_measure_mxf8f6f4_peak(4096)
    mx8_peak = moe.moe_measure_mxf8f6f4_peak(4096) if fp4 else mx_peak
    mma_name = ("tcgen05.mma kind::mxf4.block_scale (E2M1 x E2M1, M=128 N=256 K=64) on every SM (moe_measure_mxf4_peak)"
                if fp4 else "tcgen05.mma kind::mxf8f6f4.block_scale (E4M3 x E2M1, M=128 N=256 K=32) on every SM "
                "(moe_measure_mxf8f6f4_peak)")

    def finish(rec):
        if fp4 and rec["layer_roofline"]["bound"] == "tensor":
            lr = rec["layer_roofline"]
            lr["frac_of_3x_mxf8f6f4_peak"] = lr["achieved"] / (3 * mx8_peak)
            rec["roofline"]["frac_of_3x_mxf8f6f4_peak"] = rec["roofline"]["achieved"] / (3 * mx8_peak)
        return rec

    rec = finish(measure_layer(args, wl, inp, dev, world, rank, mx_peak, mma_name,
                               0 if args.no_cpu_baseline else args.cpu_seconds, True))
    others = {}
    names = [] if args.workloads == "none" or world > 1 or args.experts or args.tokens else (
        [n for n in ALL_WORKLOADS if n != wl.name] if args.workloads == "all" else
        [n for n in args.workloads.split(",") if n and n != wl.name])
    for name in names:
        owl = synth.WORKLOADS[name]
        if (owl.E, owl.d, owl.f) == (wl.E, wl.d, wl.f):  # the same expert weights: draw only x and the router
            oinp = synth.gen_layer(owl, args.seed, with_shared=False, experts=inp.experts)
            oinp.shared = inp.shared
        else:
            oinp = synth.gen_layer(owl, args.seed)
        torch.cuda.empty_cache()
        others[name] = finish(measure_layer(args, owl, oinp, dev, world, rank, mx_peak, mma_name,
                                            0 if args.no_cpu_baseline else args.cpu_seconds_other, False))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4 x mxfp4 -> f32" if fp4 else "mxfp4 x mxfp8 -> f32",
        "data": "synthetic",
    }
    line.update({k: v for k, v in rec.items() if k not in ("ms_per_step", "value", "unit")})
    if fp4:
        line["mxf8f6f4_peak_tflops"] = mx8_peak
    if others:
        line["workloads"] = {wl.name: {"ms_per_step": rec["ms_per_step"], "tokens_per_s": rec["value"],
                                       "note": "the headline above"}}
        for name, r in others.items():
            line["workloads"][name] = dict({"ms_per_step": r["ms_per_step"], "tokens_per_s": r["value"]},
                                           **{k: v for k, v in r.items() if k not in ("ms_per_step", "value", "unit",
                                                                                       "stage_timing")})
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_stack(args, wl):
    """A stack of MoE layers with every layer's experts resident: the whole model's MoE part in the decode /
    verify regime.  One canonical expert set is drawn on the host and uploaded once; each layer packs its
    own resident copy (the bytes each layer streams are what count), with its own router weights or hash
    table.  Times graph replay and direct launches; prints one JSON line."""
    import dataclasses

    import numpy as np
    import torch

    import __graft_entry__ as g
    import synth
    g.build()
    import block_scaled_fp4_sqrt_gb300 as moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L, n_hash = args.layers, min(args.hash_layers, args.layers)
    per_layer = expert_bytes(wl) * wl.E + expert_bytes(wl)  # routed + shared resident bytes per layer
    free = torch.cuda.mem_get_info(dev)[0]
    if L * per_layer > 0.9 * free:
        raise SystemExit(f"{L} layers need {L * per_layer / 1e9:.1f} GB of resident experts; {free / 1e9:.1f} GB free")
    ex = synth.gen_experts(args.seed, wl.E, wl.d, wl.f)
    sh = synth.gen_experts(args.seed, 1, wl.d, wl.f, shared=True)
    dex = moe.DeviceExperts(*(torch.from_numpy(getattr(ex, n)).to(dev) for n in ("w13", "s13", "w2", "s2")))
    dsh = moe.DeviceExperts(*(torch.from_numpy(getattr(sh, n)).to(dev) for n in ("w13", "s13", "w2", "s2")))
    V = 131072
    tok = torch.from_numpy(synth.gen_token_ids(args.seed, wl.T, V)).to(dev)
    layers = []
    for l in range(L):
        if l < n_hash:
            tab = torch.from_numpy(synth.gen_hash_table(args.seed + l, V, wl.E, wl.k)).to(dev)
            layers.append(moe.MoELayer(wl.d, wl.f, wl.E, wl.k, dex, dsh, None, None, tab, wl.T, wl.route_scale,
                                       wl.swiglu_limit, dev, args.act))
        else:
            rw, rb, _ = synth.gen_router(args.seed + l, wl.E, wl.d, wl.n_hot, wl.hot_bias)
            layers.append(moe.MoELayer(wl.d, wl.f, wl.E, wl.k, dex, dsh, torch.from_numpy(rw).to(dev),
                                       torch.from_numpy(rb).to(dev), None, wl.T, wl.route_scale, wl.swiglu_limit, dev,
                                       args.act, resident_router=True))
        layers[-1].workspace = None  # the stacks below give every layer one shared workspace
    del dex, dsh
    torch.cuda.empty_cache()
    x = torch.from_numpy(synth.gen_x(args.seed, wl.T, wl.d).view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def time_stack(use_graph):
        st = moe.MoEStack(layers, max_T=wl.T, use_graph=use_graph)
        for _ in range(max(args.warmup, 3)):
            st.forward(x, token_ids=tok, out=out)
        torch.cuda.synchronize()
        st.check()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            st.forward(x, token_ids=tok, out=out)
        e1.record(stream)
        torch.cuda.synchronize()
        st.check()
        return e0.elapsed_time(e1) / args.steps, st

    ms_direct, st_d = time_stack(False)
    st_d.close()
    cvd = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(cvd[0] if cvd else 0)
    clocks.start()
    ms_graph, st_g = time_stack(True)
    clk = clocks.stop()
    st_g.close()
    # experts each layer touched: one more pass with a workspace per layer keeps every layer's routing
    st_r = moe.MoEStack(layers, max_T=wl.T, use_graph=False, separate_workspaces=True)
    st_r.forward(x, token_ids=tok, out=out)
    torch.cuda.synchronize()
    touched = [int(torch.unique(ly.last_routing()[0]).numel()) + 1 for ly in layers]
    st_r.close()
    del st_r
    hl = dataclasses.replace(wl, hash_vocab=V)
    stack_bytes = sum(layer_bytes(hl if l < n_hash else wl, touched[l]) for l in range(L))
    pk = peaks()
    line = {
        "metric": f"MoE stack tokens/sec ({L} layers, {n_hash} hash-routed; x_(l+1) = x_l + MoE_l(x_l))",
        "value": wl.T / (ms_graph * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_graph, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4 x mxfp4 -> f32" if args.act == "mxfp4" else "mxfp4 x mxfp8 -> f32", "data": "synthetic",
        "config": dict(workload_config(wl, args.act), layers=L, hash_layers=n_hash, graph=True,
                       resident_expert_gb=round(L * per_layer / 1e9, 1)),
        "per_layer_us": ms_graph * 1e3 / L,
        "direct_launches": {"ms_per_step": ms_direct, "per_layer_us": ms_direct * 1e3 / L},
        "stack_roofline": {"bound": "hbm", "algorithmic_bytes": stack_bytes, "achieved": stack_bytes / (ms_graph * 1e-3) / 1e9,
                           "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": stack_bytes / (ms_graph * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "touched_experts_per_layer": {"min": min(touched), "max": max(touched)},
        "gpu_launches": ((L - n_hash) * layer_launches(wl) + n_hash * layer_launches(hl)) * args.steps,
        "clocks": clk,
    }
    for ly in layers:
        ly.close()
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    import synth
    if args.workload not in synth.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(synth.WORKLOADS)}")
    wl = synth.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        import dataclasses
        E = args.experts or wl.E
        T = args.tokens or wl.T
        wl = dataclasses.replace(wl, name=f"{wl.name}-E{E}-T{T}", E=E, T=T)
    if args.impl == "reference":
        import __graft_entry__ as g
        g.build_cpu()
        run_reference(args, wl)
    elif args.layers > 1:
        run_stack(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
