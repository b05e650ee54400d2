#!/usr/bin/env python
"""Throughput of the routed FP8 block-scaled MoE layer on GB300 (one JSON line on stdout).

A step is one pass of the whole layer -- moe_fp8_route_forward: routing, then prepare,
gate/up + SiLU*up requantisation, down, combine -- over one batch of synthetic tokens. The default
workload is decode: hidden 2048, intermediate 768, 128 experts, top-8 renormalised, one
token per step, stepping through 10,000 seeded tokens; the same line carries a "prefill"
record (M=4096, same shapes), the metric's tensor-bound half. Other workloads
(--workload): verify, verify_skewed (M=12), wide (M=1..64, h6144/i768/e128/top4),
wide_mxfp4 (the same shape with MXFP4 expert weights: moe_mxfp4_route_forward), prefill,
prefill_zipf (M=4096).

value   tokens/s with inputs resident in HBM: exactly --steps steps timed with CUDA events
        around CUDA-graph replays; 8 weight replicas (decode/verify/wide) or 2 (prefill)
        are rotated step by step so that no step reuses L2-resident weights. Clocks are
        sampled during about a second of untimed replays of the same steps and the timed
        region after them.
e2e     the same metric through the public API with host buffers: per step one
        moe_fp8_route_forward_pinned call -- the kernels read the hidden rows from and write
        the output to pinned host memory, route and forward enqueued by one call -- all
        inside the timed region (the Zipf workload, whose routing is given, uses a host copy,
        moe_route, moe_fp8_forward and a copy back).
roofline the dominant kernel (gate/up, the launch the step makes; at few routed rows it also
        prefetches the routed experts' w2 into L2, and those bytes count) timed alone with
        CUDA events on its stream, its algorithmic bytes (or FLOPs) per launch divided by the
        mean launch time; `direct` is the same kernel without the prefetch.
cpu_baseline the oracle (plain C++ on the host cores) on a bounded sample of the same
        workload (rank 0, N=1 only).

--impl reference times that oracle as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload on its own tokens
(the layer is data-parallel over tokens; no collective on the data path); value sums the
ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; achieved HBM GB/s (decode) / FP8 TFLOP/s (prefill)"

WORKLOADS = {
    "decode": dict(cfg="decode", M=1, desc="decode M=1: h2048 i768 e128 top-8 renormalised, "
                                          "1 token per step over 10k seeded tokens"),
    "verify": dict(cfg="verify", M=12, desc="speculative verify M=12: h2048 i768 e128 top-8"),
    "verify_skewed": dict(cfg="verify_skewed", M=12,
                          desc="speculative verify M=12, +3.0 logit bias on experts 0-3"),
    "wide": dict(cfg="wide", M=64, desc="wide expert: h6144 i768 e128 top-4"),
    "prefill": dict(cfg="prefill", M=4096, desc="prefill M=4096: h2048 i768 e128 top-8, "
                                                "router logits ~N(0,1)"),
    "prefill_zipf": dict(cfg="prefill_zipf", M=4096,
                         desc="prefill M=4096: h2048 i768 e128 top-8, Zipf(1.1) expert load"),
    "wide_mxfp4": dict(cfg="wide_mxfp4", M=64, desc="wide expert, MXFP4 weights (E2M1 codes, UE8M0 scale per 32): "
                                                   "h6144 i768 e128 top-4"),
}


def is_mx(cfg):
    return cfg.endswith("_mxfp4")


# routed rows up to which moe_fp8_forward runs the two pair kernels
PAIR_ROWS = 64
SORT_BLOCK = 256  # routed pairs one sort block covers


def launches_per_step(M, K, H, E, two_op=False):
    """Our kernels per step (FP8 and MXFP4 alike): route, gate/up, down+combine up to PAIR_ROWS
    routed rows; up to SORT_BLOCK, route, the one-launch sort (quantise, sort, gather), gate/up,
    down, combine; beyond, route, count+quantise, scatter, gather, gate/up, down, combine (the
    verify profile's producer and reducer, `two_op`, are the same five launches)."""
    R = M * K
    return 3 if R <= PAIR_ROWS else (5 if R <= SORT_BLOCK else 7)


def verify_profile(M, H, I, E, K):
    """The batch and shape the two-operation verify entry points are compiled for."""
    return (M, H, I, E, K) == (12, 2048, 768, 128, 8)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    p.add_argument("--m", type=int, default=None, help="tokens per step (wide sweep)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-threads", type=int, default=None, metavar="N",
                   help="host threads for the oracle (reference arm and cpu_baseline); default all")
    p.add_argument("--dominant-only", type=int, default=0, metavar="N",
                   help="run only N launches of the dominant kernel (gate/up, as the step launches it) and exit, "
                        "for ncu")
    p.add_argument("--dominant-direct", action="store_true",
                   help="with --dominant-only at few routed rows: the FP8 gate/up kernel without the w2 prefetch")
    p.add_argument("--profile-steps", type=int, default=0, metavar="N",
                   help="run N eager steps of the workload after 3 warm-up steps and exit, for a profiler's "
                        "launch list")
    p.add_argument("--no-verify", action="store_true",
                   help="leave the verify M=12 record out of the decode line")
    p.add_argument("--verify-route-forward", action="store_true",
                   help="verify workloads through moe_fp8_route_forward instead of the two verify operations "
                        "(moe_fp8_verify_produce + moe_fp8_verify_reduce; the same kernels)")
    p.add_argument("--no-prefill", action="store_true",
                   help="decode only: leave out the prefill record of the same line")
    p.add_argument("--clock-soak", type=float, default=1.0, metavar="S",
                   help="seconds of untimed replays before the timed region while clocks are sampled")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers
def per_expert_bytes(H, I, mx=False):
    """Weight bytes of one expert: FP8 codes + FP32 scales per 128x128 block, or MXFP4 codes
    (half a byte each) + one UE8M0 byte per 32 elements."""
    if mx:
        return 2 * I * H // 2 + 2 * I * H // 32, H * I // 2 + H * I // 32
    w13 = 2 * I * H + (2 * I // 128) * (H // 128) * 4
    w2 = H * I + (H // 128) * (I // 128) * 4
    return w13, w2


def algorithmic(H, I, E, K, M, distinct, mx=False):
    """Bytes and FLOPs one step must move / do at minimum."""
    w13, w2 = per_expert_bytes(H, I, mx)
    R = M * K
    byts = distinct * (w13 + w2) + H * E * 2 + M * H * 2 * 2 + M * K * 8
    flops = 2 * M * H * E + 6 * H * I * R
    gateup_bytes = distinct * w13 + M * H + M * (H // 128) * 4 + R * I + R * (I // 128) * 4
    gateup_flops = 4 * H * I * R
    return byts, flops, gateup_bytes, gateup_flops


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash(files=None):
    """Hash of the kernel sources (all of csrc, or the named files there)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_block_scaled_router_gb300", "csrc")
    names = sorted(files) if files else sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    for n in names:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, M=None):
    """DRAM bytes per launch from a committed ncu summary, if the sources of that kernel
    (the files the record lists) are unchanged since the counters were taken and the record
    was taken at this token count (when it names one)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        rec = d.get(workload, {}).get(kernel)
        if rec and "M" in rec and M is not None and rec["M"] != M:
            return None
        if rec and rec.get("source_hash") == kernel_source_hash(rec.get("source_files")):
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = bus_id
        self.rows = []
        self.proc = None
        self.err = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.bus_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # no nvidia-smi
            self.err = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:
            time.sleep(0.02)
        self.rows.clear()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = list(self.rows)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- oracle arm
def oracle_tokens_per_s(x, M, budget_s=15.0, max_tokens=None, threads=None):
    """Time the oracle (route + FFN) on a bounded sample of tokens on `threads` host cores
    (default: all the process may use)."""
    import oracle
    cores = threads or len(os.sched_getaffinity(0))
    K = x.shape.top_k
    total = x.hidden.shape[0]

    mx = x.w13.shape[2] * 2 == x.shape.hidden  # packed E2M1 weights

    def run(n):
        hid = x.hidden[:n]
        t0 = time.perf_counter()
        if x.ids is not None:
            ids, w = x.ids[:n], x.weights[:n]
        else:
            ids, w = oracle.route(hid, x.router_w, x.bias, K)
        if mx:
            oracle.mxfp4_forward(hid, ids, w, x.w13, x.s13, x.w2, x.s2, nthreads=cores)
        else:
            oracle.moe_forward(hid, ids, w, x.w13, x.s13, x.w2, x.s2, nthreads=cores)
        return time.perf_counter() - t0

    n = min(cores, total)
    dt = run(n)
    per_tok = dt / n
    n2 = int(min(total, max(n, budget_s / max(per_tok, 1e-9))))
    if max_tokens:
        n2 = min(n2, max_tokens)
    if n2 > n:
        n, dt = n2, run(n2)
    return n / dt, cores, n, dt


def reference_arm(args, wl, world, rank):
    if rank != 0:
        return
    from fp8_block_scaled_router_gb300 import inputs
    import oracle
    oracle.build()
    M = args.m or wl["M"]
    if is_mx(wl["cfg"]):
        x = inputs.make_mx(wl["cfg"], M=M, tokens=M)
    else:
        x = inputs.make(wl["cfg"], tokens=10000 if wl["cfg"] == "decode" else None,
                        M=M if wl["cfg"] == "wide" else None)
    steps = args.steps or 3
    warm = args.warmup if args.warmup is not None else 1
    tps, cores, n, dt = oracle_tokens_per_s(x, M, budget_s=20.0, threads=args.cpu_threads)
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": 0,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * M / tps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64-exact block sums, f32 chains",
            "data": "synthetic",
            "config": {"workload": wl["desc"], "M": M, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} tokens of the workload (route + expert FFN), "
                                       f"{dt:.1f} s, std::thread over tokens"},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def run_workload(args, wl, steps, warm, world, rank, dist, want_cpu, cpu_budget_s):
    """Measure one workload; returns its record (the JSON line's fields)."""
    import torch
    from fp8_block_scaled_router_gb300 import _lib as L
    from fp8_block_scaled_router_gb300 import inputs
    from fp8_block_scaled_router_gb300 import replicas

    cfg = wl["cfg"]
    decode = cfg == "decode"
    mx = is_mx(cfg)
    M = args.m if (args.m and cfg in ("wide", "wide_mxfp4")) else wl["M"]
    prefill = M >= 1024
    ntok = 10000 if decode else M
    if mx:
        x = inputs.make_mx(cfg, M=M, tokens=M)
    else:
        x = inputs.make(cfg, tokens=ntok if decode else None, M=M if cfg == "wide" else None)
    H, I, E, K = x.shape.hidden, x.shape.inter, x.shape.num_experts, x.shape.top_k
    # each rank steps through its own token stream (a different slice of the seeded rows)
    if decode and world > 1:
        x.hidden = np.roll(x.hidden, -replicas.token_offset(rank, world, ntok), axis=0)

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    n_rep = 2 if prefill else 8
    w13_0, s13_0, w2_0, s2_0 = dev(x.w13), dev(x.s13), dev(x.w2), dev(x.s2)
    reps = [(w13_0, s13_0, w2_0, s2_0)] + [(w13_0.clone(), s13_0.clone(), w2_0.clone(), s2_0.clone())
                                           for _ in range(n_rep - 1)]
    router = dev(x.router_w)
    bias = None if x.bias is None else dev(x.bias)
    shape = L.make_shape(H, I, E, K, M)
    ws = torch.empty(L.moe_fp8_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    L.moe_fp8_workspace_init(ws, shape)
    hidden_all = dev(x.hidden)                      # [ntok][H]
    nbatches = hidden_all.shape[0] // M
    given_ids = None if x.ids is None else (dev(x.ids), dev(x.weights))
    ids = torch.empty((nbatches, M, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((nbatches, M, K), dtype=torch.float32, device="cuda")
    out = torch.empty((nbatches, M, H), dtype=torch.int16, device="cuda")

    two_op = given_ids is None and verify_profile(M, H, I, E, K) and not args.verify_route_forward

    def step(i, stream=None):
        b = i % nbatches
        hid = hidden_all[b * M:(b + 1) * M]
        w13, s13, w2, s2 = reps[i % n_rep]
        if mx:                      # MXFP4 expert weights: routing + the two MXFP4 pair kernels
            L.moe_mxfp4_route_forward(hid, router, bias, M, True, w13, s13, w2, s2, out[b], ids[b], wts[b], ws,
                                      shape, stream=stream)
        elif two_op:                # the verify profile's two operations: producer, route reducer
            L.moe_fp8_verify_produce(hid, router, bias, M, True, w13, s13, w2, s2, ids[b], wts[b], ws, shape,
                                     stream=stream)
            L.moe_fp8_verify_reduce(wts[b], M, out[b], ws, shape, stream=stream)
        elif given_ids is not None:   # Zipf workload: the expert load is given, not routed
            L.moe_route(hid, router, bias, M, shape, True, ids[b], wts[b], stream=stream)
            ii, ww = given_ids
            L.moe_fp8_forward(hid, ii, ww, M, w13, s13, w2, s2, out[b], ws, shape, stream=stream)
        else:                       # the public one-call layer: routing + expert FFN
            L.moe_fp8_route_forward(hid, router, bias, M, True, w13, s13, w2, s2, out[b], ids[b], wts[b], ws,
                                    shape, stream=stream)

    kernels_per_step = launches_per_step(M, K, H, E, two_op)

    # distinct experts per step (accounting only)
    for i in range(min(nbatches, 64)):
        step(i)
    torch.cuda.synchronize()
    src = given_ids[0] if given_ids is not None else ids
    sample = src.reshape(-1, M * K)[: min(nbatches, 64)].cpu().numpy() if given_ids is None else \
        src.reshape(1, -1).cpu().numpy()
    distinct = float(np.mean([len(np.unique(r)) for r in sample]))
    alg_bytes, alg_flops, gu_bytes, gu_flops = algorithmic(H, I, E, K, M, distinct, mx)

    # ---- CUDA graphs: exactly `steps` steps are timed -- `full` replays of a G-step graph
    # (rotating over a few graphs so that consecutive replays walk different tokens) and one
    # graph of the remaining steps
    G = min(steps, 500 if decode else (50 if M <= 64 else 1))
    full, rem = divmod(steps, G)
    n_graphs = max(1, min(20, nbatches // G)) if decode else 1
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(s):
        for gi in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for j in range(G):
                    step(gi * G + j)
            graphs.append(g)
        g_rem = None
        if rem:
            g_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rem, stream=s):
                for j in range(rem):
                    step(full * G + j)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in range(max(1, -(-warm // G))):       # >= warm untimed steps
        graphs[i % n_graphs].replay()
    torch.cuda.synchronize()

    def replay_timed():
        for i in range(full):
            graphs[i % n_graphs].replay()
        if g_rem is not None:
            g_rem.replay()

    # clocks are sampled while the same steps run for about a second before the timed region
    # and during it (a timed region of a few steps is shorter than the sampling period)
    sampler = ClockSampler(gpu_selector(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
    t_soak = time.perf_counter()
    n_soak = 0
    while time.perf_counter() - t_soak < args.clock_soak:
        replay_timed()
        n_soak += 1
        if n_soak % 8 == 0:
            torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    ev0.record()
    replay_timed()
    ev1.record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    elapsed = ev0.elapsed_time(ev1) / 1e3
    clocks = sampler.stop() if sampler else None
    if dist:
        elapsed = replicas.slowest(elapsed, dist, "cuda")
        dist.barrier()
    value = replicas.throughput(world, steps, M, elapsed)
    ms_per_step = 1e3 * elapsed / steps

    # the dominant kernel: gate/up as the step launches it
    w2_step = distinct * per_expert_bytes(H, I, mx)[1]
    roof = dominant_kernel(L, torch, args, M, K, nbatches, hidden_all, reps, n_rep, given_ids, ids, ws, shape,
                           prefill, gu_bytes, gu_flops, mx, w2_bytes=w2_step)
    roof["traffic"] = recorded_traffic(roof["kernel"], "prefill" if prefill else cfg, M)
    if M * K <= PAIR_ROWS and not mx:  # the same kernel without the prefetch, for reference
        dr = dominant_kernel(L, torch, args, M, K, nbatches, hidden_all, reps, n_rep, given_ids, ids, ws, shape,
                             prefill, gu_bytes, gu_flops, mx, direct=True)
        roof["direct"] = {k: dr[k] for k in ("kernel", "achieved", "frac", "alg_per_launch", "mean_launch_us")}
        roof["direct"]["traffic"] = recorded_traffic("gate_up", cfg, M)

    # ---- end to end through the public API with host buffers
    e2e_steps = min(steps * max(1, n_soak), 3000 if decode else (500 if M <= 64 else 10))
    host_in = torch.empty((nbatches, M, H), dtype=torch.int16).pin_memory()
    host_in.copy_(hidden_all.view(nbatches, M, H).cpu())
    host_out = torch.empty((nbatches, M, H), dtype=torch.int16).pin_memory()
    stage = torch.empty((2, M, H), dtype=torch.int16, device="cuda")
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    cs = torch.cuda.current_stream()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for i in range(e2e_steps):
        b = i % nbatches
        w13, s13, w2, s2 = reps[i % n_rep]
        if two_op:
            hid = stage[i % 2]
            hid.copy_(host_in[b], non_blocking=True)
            L.moe_fp8_verify_produce(hid, router, bias, M, True, w13, s13, w2, s2, ids[b], wts[b], ws, shape,
                                     stream=cs)
            L.moe_fp8_verify_reduce(wts[b], M, out[b], ws, shape, stream=cs)
            host_out[b].copy_(out[b], non_blocking=True)
            continue
        if mx:  # host copy in, the one-call MXFP4 layer, copy back
            hid = stage[i % 2]
            hid.copy_(host_in[b], non_blocking=True)
            L.moe_mxfp4_route_forward(hid, router, bias, M, True, w13, s13, w2, s2, out[b], ids[b], wts[b], ws, shape,
                                      stream=cs)
            host_out[b].copy_(out[b], non_blocking=True)
            continue
        if given_ids is None:
            # the public host-buffer call: hidden read from and out written to pinned host
            # memory by the kernels, route + forward, enqueued by one call
            L.moe_fp8_route_forward_pinned(host_in[b], host_out[b], M, router, bias, True, w13, s13, w2, s2,
                                           ws, shape, stream=cs)
            continue
        hid = stage[i % 2]
        hid.copy_(host_in[b], non_blocking=True)
        L.moe_route(hid, router, bias, M, shape, True, ids[b], wts[b], stream=cs)
        ii, ww = given_ids
        L.moe_fp8_forward(hid, ii, ww, M, w13, s13, w2, s2, out[b], ws, shape, stream=cs)
        host_out[b].copy_(out[b], non_blocking=True)
    a1.record()
    torch.cuda.synchronize()
    e2e_t = a0.elapsed_time(a1) / 1e3
    if dist:
        e2e_t = replicas.slowest(e2e_t, dist, "cuda")
    e2e = {"value": replicas.throughput(world, e2e_steps, M, e2e_t), "unit": "tokens/s",
           "h2d_bytes_per_step": M * H * 2, "d2h_bytes_per_step": M * H * 2, "steps": e2e_steps}

    cpu = None
    if want_cpu:
        tps, cores, n, dt = oracle_tokens_per_s(x, M, budget_s=cpu_budget_s, threads=args.cpu_threads)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} tokens of the same workload (route + expert FFN), {dt:.1f} s, "
                         f"std::thread over tokens"}
    rec = {"value": value, "unit": "tokens/s", "steps": steps, "warmup": warm, "ms_per_step": ms_per_step,
           "config": {"workload": wl["desc"], "M": M, "hidden": H, "inter": I, "experts": E, "top_k": K,
                      "entry": ("moe_mxfp4_route_forward" if mx else
                                "moe_fp8_verify_produce + moe_fp8_verify_reduce" if two_op else
                                "moe_route + moe_fp8_forward (ids given)" if given_ids is not None else
                                "moe_fp8_route_forward"),
                      "distinct_experts_per_step": distinct,
                      "l2": f"inputs larger than L2: {n_rep} weight replicas "
                            f"({n_rep * (x.w13.nbytes + x.w2.nbytes) / 1e9:.2f} GB) rotated per step",
                      "timing": f"{steps} steps timed as {full} replays of a {G}-step CUDA graph"
                                f"{f' + one {rem}-step graph' if rem else ''}, events; wall {t_wall:.4f} s; "
                                f"{n_soak} untimed replays of the same steps before it while clocks were sampled"},
           "achieved_gbs": alg_bytes * steps / elapsed / 1e9 * world,
           "achieved_tflops": alg_flops * steps / elapsed / 1e12 * world,
           "alg_bytes_per_step": alg_bytes, "alg_flops_per_step": alg_flops,
           "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": kernels_per_step * steps,
           "clocks": clocks}
    del reps, w13_0, s13_0, w2_0, s2_0, hidden_all, ws
    torch.cuda.empty_cache()
    return rec


def dominant_kernel(L, torch, args, M, K, nbatches, hidden_all, reps, n_rep, given_ids, ids, ws, shape, prefill,
                    gu_bytes, gu_flops, mx=False, w2_bytes=0, direct=False):
    """gate/up alone, back to back in a CUDA graph on its own stream, rotating weight replicas
    and the steps' expert sets: the same launch the step makes (FP8, few routed rows: the
    gate/up kernel with the routed experts' w2 L2 prefetch, whose bytes count; otherwise the
    stage kernel after one prepare). `direct`: the FP8 few-row kernel without the prefetch."""
    pair_mode = M * K <= PAIR_ROWS
    prefetch = pair_mode and not mx and not direct
    n_k = 200 if (pair_mode or mx) else 10
    ks = torch.cuda.Stream()
    ks.wait_stream(torch.cuda.current_stream())

    def gu(i, st):
        b = i % nbatches
        hid = hidden_all[b * M:(b + 1) * M]
        w13, s13, w2, s2 = reps[i % n_rep]
        ii = given_ids[0] if given_ids is not None else ids[b]
        if prefetch:
            L.moe_fp8_gate_up_prefetch(hid, ii, M, w13, s13, w2, s2, ws, shape, stream=st)
        elif mx and M * K <= PAIR_ROWS:
            L.moe_mxfp4_gate_up_direct(hid, ii, M, w13, s13, ws, shape, stream=st)
        elif mx:
            L.moe_mxfp4_gate_up(w13, s13, M, ws, shape, stream=st)
        elif pair_mode:
            L.moe_fp8_gate_up_direct(hid, ii, M, w13, s13, ws, shape, stream=st)
        else:
            L.moe_fp8_gate_up(w13, s13, M, ws, shape, stream=st)

    with torch.cuda.stream(ks):
        if not pair_mode:  # the stage kernels read the sort of one step
            ii0 = given_ids[0] if given_ids is not None else ids[0]
            L.moe_fp8_prepare(hidden_all[:M], ii0, M, ws, shape, stream=ks)
        gu(0, ks)
        kg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kg, stream=ks):
            for i in range(n_k):
                gu(i, ks)
        kg.replay()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(ks)
        for _ in range(3):
            kg.replay()
        k1.record(ks)
    ks.synchronize()
    t_gu = k0.elapsed_time(k1) / 1e3 / (3 * n_k)
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    if prefill:
        fp8_peak = 2.0 * bf16  # FP8 dense rate = 2x the measured bf16 rate (nominal ratio)
        roof = {"bound": "tensor", "kernel": "gate_up", "achieved": gu_flops / t_gu / 1e12,
                "peak": fp8_peak, "unit": "TFLOP/s", "frac": gu_flops / t_gu / 1e12 / fp8_peak,
                "peak_source": f"{peak_src} bf16 x 2 (fp8/bf16 nominal ratio), burst"}
    else:
        nbytes = gu_bytes + (w2_bytes if prefetch else 0)
        roof = {"bound": "hbm", "kernel": "gate_up" + (" (+ w2 L2 prefetch)" if prefetch else ""),
                "achieved": nbytes / t_gu / 1e9, "peak": hbm, "unit": "GB/s", "frac": nbytes / t_gu / 1e9 / hbm,
                "peak_source": f"{peak_src} hbm_gbs"}
        gu_bytes = nbytes
    roof["alg_per_launch"] = gu_flops if prefill else gu_bytes
    roof["mean_launch_us"] = t_gu * 1e6
    return roof


def gpu_selector(torch):
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = str(getattr(props, "uuid", ""))
    return ("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or str(torch.cuda.current_device())


def ours_arm(args, wl, world, rank, local):
    import torch
    from fp8_block_scaled_router_gb300 import build as B

    B.build()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    decode = wl["cfg"] == "decode"
    M = args.m or wl["M"]
    steps = args.steps or (50000 if decode else (2000 if M <= 64 else 200))
    warm = max(3, args.warmup if args.warmup is not None else (200 if decode else 5))
    if args.dominant_only:
        dominant_only(args, wl)
        return
    if args.profile_steps:
        profile_steps(args, wl)
        return
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    rec = run_workload(args, wl, steps, warm, world, rank, dist, want_cpu, 12.0)
    # the metric's other half: prefill (M=4096) in the same run and the same line
    pre = ver = None
    if args.workload == "decode" and not args.no_verify:
        vsteps = args.steps or 20000
        ver = run_workload(args, WORKLOADS["verify"], vsteps, max(3, warm), world, rank, dist, want_cpu, 8.0)
    if args.workload == "decode" and not args.no_prefill:
        psteps = args.steps or 2500
        pre = run_workload(args, WORKLOADS["prefill"], psteps, max(3, warm), world, rank, dist, want_cpu, 12.0)
    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": steps, "warmup": warm, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": ("mxfp4 weights (e2m1 + ue8m0 per 32), fp8_e4m3 activations, f32 accumulate"
                          if is_mx(wl["cfg"]) else "fp8_e4m3 (f32 accumulate)"),
                "data": "synthetic"}
        line.update({k: v for k, v in rec.items() if k not in ("value", "unit", "steps", "warmup", "ms_per_step")})
        if ver is not None:
            line["verify"] = ver
        if pre is not None:
            line["prefill"] = pre
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def profile_steps(args, wl):
    """3 warm-up steps, then N eager steps of the workload (the launches a profiler lists)."""
    import torch
    from fp8_block_scaled_router_gb300 import _lib as L
    from fp8_block_scaled_router_gb300 import inputs

    cfg = wl["cfg"]
    mx = is_mx(cfg)
    M = args.m if (args.m and cfg in ("wide", "wide_mxfp4")) else wl["M"]
    n = 3 + args.profile_steps
    if mx:
        x = inputs.make_mx(cfg, M=M, tokens=M)
    else:
        x = inputs.make(cfg, tokens=n * M if cfg == "decode" else None, M=M if cfg == "wide" else None)
    H, I, E, K = x.shape.hidden, x.shape.inter, x.shape.num_experts, x.shape.top_k

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    reps = [(dev(x.w13), dev(x.s13), dev(x.w2), dev(x.s2)) for _ in range(2)]
    shape = L.make_shape(H, I, E, K, M)
    ws = torch.empty(L.moe_fp8_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    L.moe_fp8_workspace_init(ws, shape)
    hid_all = dev(x.hidden)
    router = dev(x.router_w)
    bias = None if x.bias is None else dev(x.bias)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    w = torch.empty((M, K), dtype=torch.float32, device="cuda")
    out = torch.empty((M, H), dtype=torch.int16, device="cuda")
    two_op = x.ids is None and verify_profile(M, H, I, E, K) and not args.verify_route_forward
    for i in range(n):
        b = i % (hid_all.shape[0] // M)
        hid = hid_all[b * M:(b + 1) * M]
        w13, s13, w2, s2 = reps[i % 2]
        if mx:
            L.moe_mxfp4_route_forward(hid, router, bias, M, True, w13, s13, w2, s2, out, ids, w, ws, shape)
        elif two_op:
            L.moe_fp8_verify_produce(hid, router, bias, M, True, w13, s13, w2, s2, ids, w, ws, shape)
            L.moe_fp8_verify_reduce(w, M, out, ws, shape)
        elif x.ids is not None:
            L.moe_route(hid, router, bias, M, shape, True, ids, w)
            L.moe_fp8_forward(hid, dev(x.ids), dev(x.weights), M, w13, s13, w2, s2, out, ws, shape)
        else:
            L.moe_fp8_route_forward(hid, router, bias, M, True, w13, s13, w2, s2, out, ids, w, ws, shape)
    torch.cuda.synchronize()


def dominant_only(args, wl):
    """Only the dominant kernel (the launch the roofline times), for a profiler: the gate/up
    GEMM (few routed rows: the direct pair kernel; otherwise the grouped GEMM after one
    prepare)."""
    import torch
    from fp8_block_scaled_router_gb300 import _lib as L
    from fp8_block_scaled_router_gb300 import inputs

    cfg = wl["cfg"]
    mx = is_mx(cfg)
    M = args.m if (args.m and cfg in ("wide", "wide_mxfp4")) else wl["M"]
    if mx:
        x = inputs.make_mx(cfg, M=M, tokens=M)
    else:
        x = inputs.make(cfg, tokens=max(M, 8) if cfg == "decode" else None, M=M if cfg == "wide" else None)
    H, I, E, K = x.shape.hidden, x.shape.inter, x.shape.num_experts, x.shape.top_k

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    n_rep = 2
    reps = [(dev(x.w13), dev(x.s13), dev(x.w2), dev(x.s2)) for _ in range(n_rep)]
    shape = L.make_shape(H, I, E, K, M)
    ws = torch.empty(L.moe_fp8_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    L.moe_fp8_workspace_init(ws, shape)
    hid = dev(x.hidden[:M])
    router = dev(x.router_w)
    bias = None if x.bias is None else dev(x.bias)
    ii = torch.empty((M, K), dtype=torch.int32, device="cuda")
    w = torch.empty((M, K), dtype=torch.float32, device="cuda")
    out = torch.empty((M, H), dtype=torch.int16, device="cuda")
    if x.ids is not None:
        ii = dev(x.ids[:M])
    else:
        L.moe_route(hid, router, bias, M, shape, True, ii, w)
    if M * K > PAIR_ROWS:
        L.moe_fp8_prepare(hid, ii, M, ws, shape)
    for i in range(args.dominant_only):
        w13, s13, w2, s2 = reps[i % n_rep]
        if mx and M * K <= PAIR_ROWS:
            L.moe_mxfp4_gate_up_direct(hid, ii, M, w13, s13, ws, shape)
        elif mx:
            L.moe_mxfp4_gate_up(w13, s13, M, ws, shape)
        elif M * K <= PAIR_ROWS and not args.dominant_direct:
            L.moe_fp8_gate_up_prefetch(hid, ii, M, w13, s13, w2, s2, ws, shape)
        elif M * K <= PAIR_ROWS:
            L.moe_fp8_gate_up_direct(hid, ii, M, w13, s13, ws, shape)
        else:
            L.moe_fp8_gate_up(w13, s13, M, ws, shape)
    torch.cuda.synchronize()


def main():
    args = parse()
    world, rank, local = dist_info()
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, wl, world, rank)
    else:
        ours_arm(args, wl, world, rank, local)


if __name__ == "__main__":
    main()
