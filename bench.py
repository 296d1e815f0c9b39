"""Benchmark of the k-aware MoE layer forward on GB300 (prints ONE JSON line).

A step is one pass of the whole hot path over one batch: router logits and
top-k_t (moe_route), permutation (moe_permute), grouped gate|up + SwiGLU
(moe_gate_up), grouped down (moe_down), weighted combine (moe_combine), plus
the shared expert where the workload has one, as one moe_layer_forward.
Inputs are seeded synthetic tensors already resident in HBM.  The headline
workload is the Mixtral-8x7B-shaped decode step (H 4096, 8 experts x 4
sub-experts of 3584, 64 one-token requests, k in {2,4,6,8}); its metric is
microseconds per layer.  Decode steps are timed as K layer calls in one CUDA
graph over rotating copies of the weights (the activated weights of
consecutive calls span at least 4x L2); prefill steps one per graph replay.

With no --workload the line's value is the headline workload's, and every
workload (tiny; Mixtral-8x7B-shaped decode; Qwen3-30B-A3B-shaped prefill;
Qwen3-30B-A3B-shaped decode at T = 1, 8, 64, 256, 1024; DeepSeek-V3-shaped
prefill) is run the same way, one after the other, and summarised in the
line's "workloads" object (value, roofline, realised routing, clocks, e2e).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--profile-calls N]

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the headline workload.  Under torchrun (N > 1) every rank runs an
independent replica (the layer has no exchange step); rank 0 prints.
--profile-calls N makes N untimed layer calls on one weight copy (for ncu).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MoE-layer tokens/s (prefill), µs/layer (decode), % of roofline, 1×GB300")
THROTTLE_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                 0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                 0x100: "display_clock_setting"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=None,
                   help="one workload only (default: the Mixtral-8x7B-shaped decode step as the "
                        "headline line, then every other workload into its 'workloads' object)")
    p.add_argument("--no-sweep", action="store_true",
                   help="headline workload only (no 'workloads' object)")
    p.add_argument("--profile-calls", type=int, default=0,
                   help="N > 0: no timing; build the workload's inputs (one weight copy), make N "
                        "moe_layer_forward calls and check the device status (for ncu captures)")
    p.add_argument("--T", type=int, default=None, help="override the token count")
    p.add_argument("--n-experts", type=int, default=None,
                   help="override the expert count (a smaller case of the same layer shape, "
                        "for profiler captures)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=30.0)
    p.add_argument("--path", type=int, default=0,
                   help="GEMM family: 0 auto, 1 token tiles, 2 weight-stationary (swap-AB)")
    p.add_argument("--router", default="linear", choices=["linear", "cg"],
                   help="linear: the expanded linear gate over all units (the default); "
                        "cg: the training-free proxy router (original router + gate neurons)")
    p.add_argument("--cg-r", type=int, default=8, help="gate neurons per sub-expert (--router cg)")
    p.add_argument("--k-mode", default="exact", choices=["exact", "batch_max", "coarse"],
                   help="budgets executed: each token's own (exact), the batch maximum for every "
                        "token (what uniform-k kernels run), or whole experts n_sub*ceil(k/n_sub)")
    p.add_argument("--k-normal", default=None,
                   help="MU,SIGMA: draw budgets k = clip(round(N(MU, SIGMA^2)), 1, k_max) per "
                        "token instead of the workload's uniform draw")
    p.add_argument("--fold", type=int, default=0,
                   help="decode expert-pool folding to a dynamic pool of D units (0: off)")
    p.add_argument("--tiered", action="store_true",
                   help="offline queue experiment: profile T(n, k) on this GPU, then time a "
                        "synthetic request queue batched FIFO at the batch-max budget, by "
                        "quality tiers (Eq. 5) at the batch-max budget, and FIFO at every "
                        "request's own budget")
    p.add_argument("--paths", action="store_true",
                   help="path-composed execution with source-grouped reuse: time "
                        "moe_layer_forward_paths on the seeded path recipe against the same "
                        "pipeline with diagonal paths and against moe_layer_forward")
    p.add_argument("--force-pair", action="store_true",
                   help="run grouped prefill GEMMs on the CTA-pair kernel (debug flag)")
    return p.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the slowest replica sets the job's
    time); the value itself with one rank.  Needs the default process group
    when world > 1 (NCCL on the GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: every replica processes its own batch (weak
    scaling), all of them within the slowest replica's time."""
    return tokens_per_rank * world / (ms * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int, out_path: str):
        self.path = out_path
        self.proc = None
        self.index = index

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], 0
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 5:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                reasons |= int(parts[4], 16)
            except ValueError:
                continue
        if not sm:
            return None
        names = [n for b, n in THROTTLE_BITS.items() if reasons & b and n != "gpu_idle"]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": names,
                "samples": len(sm)}


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "aware_moe_expert_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(workload_name: str, kernel: str, per_launch_units: float):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    e = table.get(f"{workload_name}:{kernel}")
    if not e or e.get("source_hash") != source_hash(*e.get("sources", ["gemm.cu"])):
        return None
    return float(e["dram_bytes_per_launch"]) * per_launch_units / float(e.get("units", per_launch_units))


def run_ours(args, wl, rank, world, local):
    import torch
    from aware_moe_expert_gb300 import binding as B
    from aware_moe_expert_gb300.inputs import make_layer_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = make_layer_inputs(wl, dev, seed=wl.seed + 1000 * rank)
    if args.k_normal is not None:
        from aware_moe_expert_gb300.inputs import draw_k_normal
        mu, sigma = (float(v) for v in args.k_normal.split(","))
        d["k_per_token"] = draw_k_normal(wl.T, mu, sigma, wl.k_max, seed=wl.seed + 9, device=dev)
    if args.k_mode != "exact":
        from aware_moe_expert_gb300.inputs import apply_k_mode
        d["k_per_token"] = apply_k_mode(d["k_per_token"], args.k_mode, wl.n_sub, wl.k_max)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    desc.path = args.path
    if args.force_pair:
        desc.debug_flags |= B.DEBUG_FORCE_PAIR
    T, H, E_r, k_max, I_sub = wl.T, wl.H, wl.E_r, wl.k_max, wl.I_sub
    cg = None
    if args.router == "cg":
        from aware_moe_expert_gb300.inputs import make_cg_inputs
        ci = make_cg_inputs(wl, dev, seed=wl.seed + 1000 * rank, r=args.cg_r)
        proxy_w = torch.empty(E_r * 2 * args.cg_r, H, dtype=torch.bfloat16, device=dev)
        st0 = torch.zeros(1, dtype=torch.int32, device=dev)
        B.check(B.moe_pack_proxy_rows(desc, args.cg_r, d["w_gate_up"], ci["gate_neurons"],
                                      proxy_w, st0), "moe_pack_proxy_rows")
        cg = B.CgRouter(m=wl.native_m, r=args.cg_r, router_w_expert=ci["router_w_expert"],
                        proxy_w=proxy_w, kappa=ci["kappa"])
    fold = None
    if args.fold > 0:
        from aware_moe_expert_gb300.inputs import make_fold_tables
        S_t, L_t = make_fold_tables(E_r, dev, seed=wl.seed + 5)
        fold = B.FoldDesc(D=args.fold, S=S_t, L=L_t)
        fidx = torch.empty(T, k_max, dtype=torch.int32, device=dev)
        fw = torch.empty(T, k_max, dtype=torch.float32, device=dev)
        fk = torch.empty(T, dtype=torch.int32, device=dev)
    ws_bytes = B.moe_workspace_size(desc) if cg is None else B.moe_cg_workspace_size(desc, cg)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    idx = torch.empty(T, k_max, dtype=torch.int32, device=dev)
    w = torch.empty(T, k_max, dtype=torch.float32, device=dev)
    counts = torch.empty(E_r, dtype=torch.int32, device=dev)
    offsets = torch.empty(E_r + 1, dtype=torch.int32, device=dev)
    st_tok = torch.empty(T * k_max, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k_max, dtype=torch.int32, device=dev)
    act = torch.empty(T * k_max, I_sub, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T * k_max, H, dtype=torch.bfloat16, device=dev)
    ysh = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if wl.I_shared else None
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def call_route(sp):
        if cg is not None:
            B.check(B.moe_route_cg(desc, cg, d["x"], d["k_per_token"], None, None, idx, w, st, ws,
                                   sp), "moe_route_cg")
            return
        B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], None, idx, w,
                            st, ws, sp), "moe_route")

    def call_fold(sp):
        B.check(B.moe_fold_decode(desc, fold, idx, w, d["k_per_token"], fidx, fw, fk, None, st,
                                  ws, sp), "moe_fold_decode")

    def call_permute(sp):
        if fold is not None:
            B.check(B.moe_permute(desc, fidx, fk, counts, offsets, st_tok, inv, st, ws, sp),
                    "moe_permute")
            return
        B.check(B.moe_permute(desc, idx, d["k_per_token"], counts, offsets, st_tok, inv, st, ws,
                              sp), "moe_permute")

    def call_shared(sp):
        B.check(B.moe_shared_ffn(desc, d["x"], ysh, st, ws, sp), "moe_shared_ffn")

    def call_gate_up(sp):
        B.check(B.moe_gate_up(desc, d["x"], st_tok, offsets, d["w_gate_up"], act, st, ws, sp),
                "moe_gate_up")

    def call_down(sp):
        B.check(B.moe_down(desc, act, offsets, d["w_down"], y, st, ws, sp), "moe_down")

    def call_grouped_ffn(sp):
        B.check(B.moe_grouped_ffn(desc, d["x"], st_tok, offsets, d["w_gate_up"], d["w_down"], y,
                                  st, ws, sp), "moe_grouped_ffn")

    def call_combine(sp):
        if fold is not None:
            B.check(B.moe_combine(desc, y, ysh, inv, fw, fk, out, st, sp), "moe_combine")
            return
        B.check(B.moe_combine(desc, y, ysh, inv, w, d["k_per_token"], out, st, sp), "moe_combine")

    calls = [("route", call_route)]
    if fold is not None:
        calls.append(("fold", call_fold))
    calls.append(("permute", call_permute))
    if ysh is not None:
        calls.append(("shared_ffn", call_shared))
    calls += [("gate_up", call_gate_up), ("down", call_down), ("grouped_ffn", call_grouped_ffn),
              ("combine", call_combine)]

    def step(sp):
        for _, f in calls:
            f(sp)

    out_fused = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws_fused = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    weight_sets = [d]     # decode: rotating copies of the weights, added below

    def layer_step(sp, c=0):
        wt = weight_sets[c]
        if fold is not None:
            B.check(B.moe_layer_forward_fold(desc, fold, d["x"], wt["router_w"], wt["w_gate_up"],
                                             wt["w_down"], d["k_per_token"], out_fused, st,
                                             ws_fused, sp), "moe_layer_forward_fold")
            return
        if cg is not None:
            B.check(B.moe_layer_forward_cg(desc, cg, d["x"], wt["w_gate_up"], wt["w_down"],
                                           d["k_per_token"], out_fused, st, ws_fused, sp),
                    "moe_layer_forward_cg")
            return
        B.check(B.moe_layer_forward(desc, d["x"], wt["router_w"], wt["w_gate_up"], wt["w_down"],
                                    d["k_per_token"], out_fused, st, ws_fused, sp),
                "moe_layer_forward")

    # one eager pass: realised routing statistics, per-device set-up
    with torch.cuda.stream(stream):
        step(sp)
        layer_step(sp)
    torch.cuda.synchronize(dev)
    code = B.moe_get_device_status(st, sp)
    if code != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(code, code)}")
    cnt = counts.cpu().numpy()
    n_assign = int(cnt.sum())
    D = int(np.count_nonzero(cnt))

    # The step is replayed from CUDA graphs so that the device timeline is
    # not stretched by host enqueue time: one graph of moe_layer_forward (the
    # whole step, the timed value) and one graph per component call (the
    # per-call breakdown and the dominant call's roofline).
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            fn(torch.cuda.current_stream().cuda_stream)
        return g
    g_parts = [(n, capture(f)) for n, f in calls]

    # L2 handling.  Decode: the K timed steps are K layer calls in one CUDA
    # graph over rotating copies of the weights, enough copies that the
    # activated weights of consecutive calls span at least 4x L2 (no flush,
    # no host launch gap between layers; time / K per layer).  Prefill: one
    # layer per graph replay, L2 flushed between steps (2x-L2 write) unless
    # the step streams far more than L2 anyway.  The per-call breakdown uses
    # the flush whenever the activated weights are below 4x L2.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    w_active = D * 3 * H * I_sub * 2 + (3 * H * wl.I_shared * 2 if wl.I_shared else 0)
    rotate = wl.phase == "decode"
    flush_parts = w_active < 4 * l2
    flush = flush_parts and not rotate
    flush_buf = (torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
                 if flush_parts else None)
    if rotate:
        keys = [k for k in ("router_w", "w_gate_up", "w_down", "w_shared_gate_up",
                            "w_shared_down") if d.get(k) is not None]
        per_copy = sum(d[k].numel() * d[k].element_size() for k in keys)
        n_copies = max(2, -(-4 * l2 // max(w_active, 1)))
        while n_copies > 2 and n_copies * per_copy > (24 << 30):
            n_copies -= 1
        for _ in range(n_copies - 1):
            weight_sets.append({k: d[k].clone() for k in keys})
    g_full = capture(layer_step)
    g_all = None
    if rotate:
        def all_steps(sp):
            for i in range(args.steps):
                layer_step(sp, i % len(weight_sets))
        g_all = capture(all_steps)

    def maybe_flush():
        if flush:
            flush_buf.zero_()

    def flush_for_parts():
        if flush_parts:
            flush_buf.zero_()

    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n_parts = len(g_parts)
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(n_parts + 1)]
           for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        if rotate:
            for _ in range(-(-args.warmup // args.steps)):
                g_all.replay()
        else:
            for _ in range(args.warmup):
                maybe_flush()
                g_full.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    import tempfile
    smi_path = os.path.join(os.environ.get("MOE_BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                            f"moe_bench_clocks_r{rank}.csv")
    os.makedirs(os.path.dirname(smi_path), exist_ok=True)
    with ClockSampler(local, smi_path) as cs:
        t_wall0 = time.perf_counter()
        with torch.cuda.stream(stream):
            if rotate:
                ev0[0].record(stream)
                g_all.replay()
                ev1[0].record(stream)
            else:
                for i in range(args.steps):
                    maybe_flush()
                    ev0[i].record(stream)
                    g_full.replay()
                    ev1[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        # per-call breakdown, same number of steps
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_for_parts()
                evp[i][0].record(stream)
                for j, (_, g) in enumerate(g_parts):
                    g.replay()
                    evp[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        # identical untimed steps so that the clock record covers >= ~1.5 s of load
        t_extra = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t_extra < 1.5:
                if rotate:
                    g_all.replay()
                else:
                    for _ in range(20):
                        maybe_flush()
                        g_full.replay()
                torch.cuda.synchronize(dev)
    code = B.moe_get_device_status(st, sp)
    if code != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(code, code)}")
    if rotate:
        step_ms = np.array([ev0[0].elapsed_time(ev1[0]) / args.steps])
    else:
        step_ms = np.array([ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)])
    ms = max_over_ranks(float(step_ms.mean()), world, dev)
    per = np.array([[evp[i][j].elapsed_time(evp[i][j + 1]) for j in range(n_parts)]
                    for i in range(args.steps)])
    parts = {n: float(per[:, j].mean() * 1000.0) for j, (n, _) in enumerate(g_parts)}
    del g_full, g_parts

    # end to end through the public call with host buffers: every step copies
    # its inputs (x, k) from pinned host memory and its output back (decode
    # steps rotate over the weight copies).  Unless L2 is flushed between
    # steps, the steps are pipelined on three streams: step i+1's
    # host->device copy and step i-1's device->host copy run on their own
    # streams while step i computes (double-buffered device tensors); the
    # timed region spans all K steps, first copy to last.  With the flush each
    # step runs copy -> layer -> copy in order and is timed alone, the flush
    # outside the timed region.
    e2e = None
    if not args.no_e2e:
        layer = B.MoeLayer(desc, dev)
        if cg is not None:
            layer.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        # a step's inputs (x, then k) sit in one pinned host buffer and are
        # copied with one host->device copy into one of two device buffers
        xb, kb = T * H * 2, T * 4
        in_bytes = (xb + 255) // 256 * 256 + kb
        hin = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        hin[:xb].copy_(d["x"].cpu().contiguous().view(torch.uint8).reshape(-1))
        hin[in_bytes - kb:].copy_(d["k_per_token"].cpu().contiguous().view(torch.uint8))
        din = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        dx = [b_[:xb].view(torch.bfloat16).view(T, H) for b_ in din]
        dk = [b_[in_bytes - kb:].view(torch.int32) for b_ in din]
        hout = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        dout = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        cdesc = desc.c()   # built once, as a serving loop would

        def forward(b, i=0):
            wt = weight_sets[i % len(weight_sets)]   # decode: the rotating copies
            if cg is not None:
                B.check(B.moe_layer_forward_cg(desc, cg, dx[b], wt["w_gate_up"], wt["w_down"],
                                               dk[b], dout[b], layer.status, layer.workspace, sp))
            else:
                B.check(B.moe_layer_forward(cdesc, dx[b], wt["router_w"], wt["w_gate_up"],
                                            wt["w_down"], dk[b], dout[b], layer.status,
                                            layer.workspace, sp))

        def run_serial(n):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n)]
            for i in range(n):
                with torch.cuda.stream(stream):
                    if flush:
                        flush_buf.zero_()
                    ev[i][0].record(stream)
                    din[0].copy_(hin, non_blocking=True)
                    forward(0, i)
                    hout[0].copy_(dout[0], non_blocking=True)
                    ev[i][1].record(stream)
            torch.cuda.synchronize(dev)
            return float(np.mean([a.elapsed_time(b) for a, b in ev]))

        def run_pipelined(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_comp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            t0.record(s_in)
            for i in range(n):
                b = i & 1
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])     # step i-2 has read dx[b], dk[b]
                with torch.cuda.stream(s_in):
                    din[b].copy_(hin, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])    # dout[b] copied out
                with torch.cuda.stream(stream):
                    forward(b, i)
                    ev_comp[i].record(stream)
                s_out.wait_event(ev_comp[i])
                with torch.cuda.stream(s_out):
                    hout[b].copy_(dout[b], non_blocking=True)
                    ev_out[i].record(s_out)
            s_out.wait_event(ev_comp[n - 1])
            t1.record(s_out)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1) / n

        # one C call per step with the host buffers (moe_layer_forward_host:
        # copy in, layer, copy out on one stream); decode steps move little
        # data, so the call's lower host cost matters more than overlapping
        # the copies
        hx = hin[:xb].view(torch.bfloat16).view(T, H)
        hk = hin[in_bytes - kb:].view(torch.int32)

        def run_host_calls(n):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            t0.record(stream)
            for i in range(n):
                wt = weight_sets[i % len(weight_sets)]
                B.check(B.moe_layer_forward_host(cdesc, hx, hk, hout[0], dx[0], dk[0], dout[0],
                                                 wt["router_w"], wt["w_gate_up"], wt["w_down"],
                                                 layer.status, layer.workspace, sp))
            t1.record(stream)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1) / n

        h2d = in_bytes
        d2h = T * H * 2
        if flush:
            run_serial(args.warmup)
            e2e_ms = run_serial(args.steps)
            e2e_mode = "serial per step (copy in, layer, copy out; L2 flushed between steps)"
        else:
            run_pipelined(max(args.warmup, 2))
            e2e_ms = run_pipelined(args.steps)
            e2e_mode = ("pipelined: step i+1's copy in and step i-1's copy out overlap step i "
                        "on two copy streams; K steps timed first copy to last")
            if wl.phase == "decode" and cg is None:
                run_host_calls(max(args.warmup, 2))
                host_ms = run_host_calls(args.steps)
                if host_ms < e2e_ms:
                    e2e_ms = host_ms
                    h2d = xb + kb
                    e2e_mode = ("one moe_layer_forward_host call per step (x and k copied in "
                                "from pinned host memory, the layer, out copied back, one "
                                "stream); K steps timed first call to last")
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        e2e = (e2e_ms, h2d, d2h, e2e_mode)
        if layer.device_status(sp) != 0:
            raise RuntimeError("device status after e2e")

    peaks = load_peaks()
    # algorithmic work (spec formulas)
    F_routed = 6.0 * H * I_sub * n_assign
    F_shared = 6.0 * H * wl.I_shared * T
    # router rows: one per unit (linear gate), or the original router's rows
    # plus the packed gate-neuron rows (proxy router)
    router_rows = E_r if cg is None else wl.n_experts + E_r * 2 * args.cg_r
    F_router = 2.0 * T * H * router_rows
    F = F_routed + F_shared + F_router
    Bytes = 2.0 * (D * 3 * H * I_sub + 3 * H * wl.I_shared + router_rows * H + 2 * T * H)
    # The bf16 peak a tensor-bound line is judged against: the burst rate
    # (cuBLAS timed alone) for steps under 1 ms, the sustained rate (cuBLAS
    # back to back for seconds, at the power cap) for longer steps, which run
    # back to back under the same cap.  Both fractions are reported.
    long_step = ms >= 1.0
    P_bf16 = peaks["bf16_tflops_sustained"] if long_step else peaks["bf16_tflops"]
    peak_kind = "sustained" if long_step else "burst"
    t_F = F / (P_bf16 * 1e12)
    t_B = Bytes / (peaks["hbm_gbs"] * 1e9)
    t_roof_us = max(t_F, t_B) * 1e6
    bound = "tensor" if t_F > t_B else "hbm"
    t_roof_burst_us = max(F / (peaks["bf16_tflops"] * 1e12), t_B) * 1e6
    t_roof_sus_us = max(F / (peaks["bf16_tflops_sustained"] * 1e12), t_B) * 1e6

    # dominant kernel.  Decode: moe_grouped_ffn, whose work is one fused
    # kernel (gate|up + SwiGLU + down) after the row gather; prefill: the
    # grouped gate|up GEMM (2/3 of the routed FLOPs).
    gu_us = parts["gate_up"]
    if wl.phase == "decode":
        ffn_us = parts["grouped_ffn"]
        alg = 2.0 * (3 * D * H * I_sub + 2 * n_assign * H)   # unit weights + x rows + y rows
        achieved = alg / (ffn_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic_for(wl.name, "grouped_ffn", 1.0),
                "kernel": "moe_grouped_ffn (row gather + fused decode FFN kernel: "
                          "gate|up + SwiGLU + down)",
                "algorithmic_bytes": alg, "peak_source": peaks["source"] + " hbm_gbs"}
    else:
        alg = 4.0 * H * I_sub * n_assign
        achieved = alg / (gu_us * 1e-6) / 1e12
        pk = P_bf16
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(achieved / pk, 4), "traffic": traffic_for(wl.name, "gate_up", 1.0),
                "kernel": "moe_gate_up (row gather + grouped gate|up GEMM, SwiGLU epilogue)",
                "algorithmic_flops": alg,
                "peak_source": peaks["source"] + (" bf16_tflops_sustained (step of 1 ms or more)"
                                                  if long_step else " bf16_tflops (burst)"),
                "frac_burst": round(achieved / peaks["bf16_tflops"], 4),
                "frac_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}

    n_launch = launches_per_step(wl, T, args.path, fold=fold is not None, cg=cg is not None) + \
        (2 if cg is not None else 0)
    us = ms * 1000.0
    res = {
        "metric": METRIC,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
    }
    if wl.phase == "decode":
        res.update({"value": round(us, 2), "unit": "µs/layer", "higher_is_better": False})
    else:
        res.update({"value": round(job_tokens_per_s(T, world, ms), 1), "unit": "tokens/s",
                    "higher_is_better": True})
    res["config"] = {"workload": wl.name, "T": T, "H": H, "experts": wl.n_experts,
                     "n_sub": wl.n_sub, "E_r": E_r, "I_sub": I_sub, "I_shared": wl.I_shared,
                     "k_choices": list(wl.k_choices), "k_per": wl.k_per, "score": wl.score,
                     "k_mode": args.k_mode, "k_normal": args.k_normal,
                     "parallelism": f"replicas{world}",
                     "fold": (None if fold is None else
                              f"decode expert-pool folding: dynamic pool of {args.fold} units, "
                              "synthetic S/L tables"),
                     "router": ("linear gate over all units" if cg is None else
                                f"proxy router: top-{wl.native_m} experts, {args.cg_r} gate "
                                f"neurons per sub-expert, even allocation table"),
                     "l2": (f"{len(weight_sets)} rotating weight copies, K layer calls in one "
                            f"CUDA graph ({len(weight_sets) * w_active / 2**20:.0f} MiB of "
                            f"activated weights across copies vs {l2 >> 20} MiB L2)" if rotate else
                            f"flushed between steps ({2 * l2 >> 20} MiB write)" if flush else
                            f"inputs larger than L2 ({w_active / 2**20:.0f} MiB of active weights "
                            f"per step vs {l2 >> 20} MiB L2)")}
    res["realised"] = {"n_assign": n_assign, "distinct_units": D, "k_mean": n_assign / T}
    res["roofline_layer"] = {"t_roof_us": round(t_roof_us, 2), "bound": bound,
                             "frac": round(t_roof_us / us, 4), "flops": F, "bytes": Bytes,
                             "bf16_peak": peak_kind,
                             "frac_burst": round(t_roof_burst_us / us, 4),
                             "frac_sustained": round(t_roof_sus_us / us, 4)}
    res["roofline"] = roof
    res["breakdown_us"] = {k: round(v, 2) for k, v in parts.items()}
    res["gpu_launches"] = n_launch * args.steps
    if e2e is not None:
        e2e_ms, h2d, d2h, e2e_mode = e2e
        if wl.phase == "decode":
            res["e2e"] = {"value": round(e2e_ms * 1000.0, 2), "unit": "µs/layer",
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode}
        else:
            res["e2e"] = {"value": round(job_tokens_per_s(T, world, e2e_ms), 1), "unit": "tokens/s",
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode}
    clocks = cs.summary()
    res["clocks"] = clocks
    res["wall_s_timed"] = round(t_wall, 4)
    return res, d


def launches_per_step(wl, T, path=0, fold=False, cg=False):
    """Kernels libmoe enqueues per moe_layer_forward (mirrors the host
    sequencing in csrc/api.cu: router + top-k (one cluster launch on CUDA
    cores, or the tensor-core GEMM and the top-k kernel), permutation (fused
    into the router launch for <= 8 tokens; above 128 tokens the top-k kernel
    also writes its bitmap), [folding], [shared expert], the fused decode FFN
    or gate|up (+ the split-K reduction of the weight-stationary family) and
    down (+ its split reduction), combine)."""
    n_cap = T * wl.k_max
    decode = path == 2 or (path == 0 and n_cap <= 64 * wl.E_r)
    budget = 256 << 20
    tc_router = T >= 128 and wl.E_r in (64, 128, 256)
    cluster_router = not tc_router and wl.H <= 12288
    decode_ffn = decode and wl.H % 128 == 0 and wl.I_sub % 128 == 0
    fused_front = cluster_router and T <= 8 and not fold   # logits + top-k + permutation (+ gather)
    if fused_front:
        n = 1
    else:
        n = 1 if cluster_router else 2               # logits (+ top-k)
        if T <= 128:
            n += 1                                   # permutation in one CTA
        else:                                        # [bitmap,] scan, scatter
            n += 2 if not (cluster_router or fold or cg) else 3
    n += 4 if fold else 0                            # fold: scores, pool, target map, remap
    n += 2 if wl.I_shared else 0                     # shared expert gate|up, down
    if decode_ffn:
        # fused decode FFN; it gathers its token rows itself inside
        # moe_layer_forward, the fold and proxy-router layers run the row gather
        n += 1 if (fused_front or not (fold or cg)) else 2
    else:
        # gate|up GEMM; the decode family reads a gathered copy of x, the
        # prefill kernel gathers its rows itself
        n += 2 if decode else 1
        if decode and wl.I_sub % 64 == 0:
            n += 1 if budget // max(n_cap * 2 * wl.I_sub * 4, 1) >= 2 else 0
        n += 1                                       # down GEMM
        if decode and wl.H % 128 == 0:
            n += 1 if budget // max(n_cap * wl.H * 4, 1) >= 2 else 0
    n += 1                                           # combine
    return n


def oracle_sample(wl, d_host, budget_s):
    """Time the fp64 oracle on a bounded sample of the workload's tokens.
    Returns (seconds, n_tokens, description)."""
    from oracle import moe_oracle as O
    T = wl.T
    spec_full = dict(H=wl.H, n_experts=wl.n_experts, n_sub=wl.n_sub, I_sub=wl.I_sub,
                     k_max=wl.k_max, score=wl.score, renorm=wl.renorm,
                     route_scale=wl.route_scale, I_shared=wl.I_shared)
    n = T if wl.phase == "decode" else min(T, 64)
    spec = O.LayerSpec(T=n, **spec_full)
    t0 = time.perf_counter()
    O.layer_forward(spec, d_host["x"][:n], d_host["router_w"], d_host["w_gate_up"],
                    d_host["w_down"], d_host["k"][:n], expert_bias=d_host["bias"],
                    w_shared_gate_up=d_host.get("sgu"), w_shared_down=d_host.get("sd"))
    dt = time.perf_counter() - t0
    return dt, n


def host_copy(d, wl):
    from aware_moe_expert_gb300.inputs import bf16_bits
    h = {"x": bf16_bits(d["x"]), "router_w": bf16_bits(d["router_w"]),
         "w_gate_up": (lambda u, w=d["w_gate_up"]: bf16_bits(w[u])),
         "w_down": (lambda u, w=d["w_down"]: bf16_bits(w[u])),
         "k": d["k_per_token"].cpu().numpy(),
         "bias": None if d["expert_bias"] is None else d["expert_bias"].cpu().numpy()}
    if wl.I_shared:
        h["sgu"] = bf16_bits(d["w_shared_gate_up"])
        h["sd"] = bf16_bits(d["w_shared_down"])
    return h


def cpu_baseline_entry(wl, d, budget_s):
    h = host_copy(d, wl)
    dt, n = oracle_sample(wl, h, budget_s)
    cores = os.cpu_count()
    if wl.phase == "decode":
        value, unit = dt * 1e6, "µs/layer"
        sample = f"the whole {wl.T}-token decode batch, one layer"
    else:
        value, unit = n / dt, "tokens/s"
        sample = f"first {n} of {wl.T} tokens (tokens are independent), one layer"
    return {"value": round(value, 3), "unit": unit, "cores": cores, "kind": "oracle",
            "sample": sample + "; float64 numpy, BLAS matmuls on all host cores, "
                      "element-wise steps single-threaded", "seconds": round(dt, 3)}


def run_reference(args, wl, rank, world):
    """--impl reference: the oracle, as it stands, timed on the host cores."""
    if rank != 0:
        return None
    import torch
    from aware_moe_expert_gb300.inputs import make_layer_inputs
    d = make_layer_inputs(wl, "cpu") if wl.T * wl.H < 1 << 26 and wl.E_r * wl.H * wl.I_sub < 1 << 31 \
        else make_layer_inputs(wl, "cpu")
    h = host_copy(d, wl)
    times = []
    for i in range(args.warmup + args.steps):
        dt, n = oracle_sample(wl, h, args.cpu_budget_s)
        if i >= args.warmup:
            times.append(dt)
        if sum(times) > 240:
            break
    dt = float(np.mean(times))
    if wl.phase == "decode":
        value, unit, hib = dt * 1e6, "µs/layer", False
        sample = f"the whole {wl.T}-token decode batch, one layer"
    else:
        value, unit, hib = n / dt, "tokens/s", True
        sample = f"first {n} of {wl.T} tokens, one layer"
    del torch
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": unit,
            "n_gpus": world, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 3), "unit": unit, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_tiered(args, wl, rank, world, local):
    """Quality-tiered batching on the prefill-shaped workload.

    1. T(n, k): moe_layer_forward with every token at budget k, n tokens,
       CUDA-event mean of timed calls with L2 flushed before each.
    2. A seeded synthetic offline queue (request sizes and budgets drawn
       uniformly) is batched three ways under the token budget M = T of the
       workload: FIFO by arrival at the batch-max budget; by quality tiers with
       Eq. (5) (moe_tier_schedule, the library's host scheduler) at the
       batch-max budget; FIFO at every request's own budget (this library's
       layer runs per-token budgets natively).  Each batch is run and timed.
    """
    import torch
    from aware_moe_expert_gb300 import binding as B
    from aware_moe_expert_gb300.inputs import make_layer_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = make_layer_inputs(wl, dev, seed=wl.seed + 1000 * rank)
    M = wl.T
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    descs, wss, outs = {}, {}, {}

    def run_batch(k_vec, reps):
        n = int(k_vec.numel())
        if n not in descs:
            descs[n] = B.desc_for(wl, T=n, expert_bias=d["expert_bias"])
            wss[n] = torch.empty(B.moe_workspace_size(descs[n]), dtype=torch.uint8, device=dev)
            outs[n] = torch.empty(n, wl.H, dtype=torch.bfloat16, device=dev)
        x = d["x"][:n]
        times = []
        with torch.cuda.stream(stream):
            for r in range(reps + 1):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                B.check(B.moe_layer_forward(descs[n], x, d["router_w"], d["w_gate_up"],
                                            d["w_down"], k_vec, outs[n], st, wss[n],
                                            stream.cuda_stream), "moe_layer_forward")
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(dev)
        return float(np.mean([a.elapsed_time(b) for a, b in times[1:]])) * 1000.0

    k_points = sorted(set(wl.k_choices))
    n_points = [M // 16, M // 8, M // 4, M // 2, M]
    t_us = [[run_batch(torch.full((n,), k, dtype=torch.int32, device=dev), 3) for n in n_points]
            for k in k_points]
    table = B.CostTable(n_points, k_points, t_us)

    rng = np.random.default_rng(wl.seed + 77)
    n_req = 64
    reqs = [(float(i), int(rng.integers(M // 64, M // 8 + 1)), int(rng.choice(k_points)))
            for i in range(n_req)]
    total_tok = sum(r[1] for r in reqs)

    def fifo(reqs_):
        out, cur, tok = [], [], 0
        for i in range(len(reqs_)):
            if cur and tok + reqs_[i][1] > M:
                out.append(cur)
                cur, tok = [], 0
            cur.append(i)
            tok += reqs_[i][1]
        if cur:
            out.append(cur)
        return out

    def time_batches(batches, batch_max):
        tot = 0.0
        for b in batches:
            if batch_max:
                kk = max(reqs[i][2] for i in b)
                ks = [kk] * sum(reqs[i][1] for i in b)
            else:
                ks = [reqs[i][2] for i in b for _ in range(reqs[i][1])]
            tot += run_batch(torch.tensor(ks, dtype=torch.int32, device=dev), 2)
        return tot

    f_batches = fifo(reqs)
    batch_of, bk, _ = B.moe_tier_schedule(reqs, M, table)
    t_batches = [[] for _ in bk]
    order = sorted(range(n_req), key=lambda i: (reqs[i][2], reqs[i][0], i))
    for i in order:
        t_batches[batch_of[i]].append(i)
    t_fifo_max = time_batches(f_batches, True)
    t_tiered = time_batches(t_batches, True)
    t_exact = time_batches(f_batches, False)
    served = lambda batches: sum(max(reqs[i][2] for i in b) * reqs[j][1]  # noqa: E731
                                 for b in batches for j in b)
    exact_assign = sum(r[1] * r[2] for r in reqs)
    return {
        "metric": "MoE-layer tokens/s over an offline request queue (quality-tiered batching)",
        "unit": "tokens/s", "higher_is_better": True, "n_gpus": world, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "token_budget_M": M, "requests": n_req,
                   "request_tokens": [M // 64, M // 8], "k_choices": k_points},
        "cost_table_us": {"n_points": n_points, "k_points": k_points,
                          "t_us": [[round(v, 2) for v in row] for row in t_us]},
        "value": round(total_tok / (t_tiered * 1e-6), 1),
        "fifo_batch_max_k": {"tokens_per_s": round(total_tok / (t_fifo_max * 1e-6), 1),
                             "batches": len(f_batches),
                             "served_assignments": served(f_batches)},
        "tiered_batch_max_k": {"tokens_per_s": round(total_tok / (t_tiered * 1e-6), 1),
                               "batches": len(t_batches),
                               "served_assignments": served(t_batches)},
        "fifo_exact_k": {"tokens_per_s": round(total_tok / (t_exact * 1e-6), 1),
                         "batches": len(f_batches), "served_assignments": exact_assign},
    }


def run_paths(args, wl, rank, world, local):
    """Path-composed execution (each path = expansion of a source unit, then
    projection of a target unit; paths of a token that share a source share
    one expansion).  Paths come from the layer's own routing through the
    seeded recipe of the input generator (consecutive slots share a source).
    Three CUDA graphs, timed the same way as the main bench: composed paths,
    the same pipeline with diagonal paths (every path its own source), and
    moe_layer_forward (routing included there, excluded from the other two)."""
    import torch
    from aware_moe_expert_gb300 import binding as B
    from aware_moe_expert_gb300.inputs import make_layer_inputs, make_paths

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = make_layer_inputs(wl, dev, seed=wl.seed + 1000 * rank)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    T, H, k_max = wl.T, wl.H, wl.k_max
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    idx = torch.empty(T, k_max, dtype=torch.int32, device=dev)
    w = torch.empty(T, k_max, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], None, idx, w, st, ws,
                        stream.cuda_stream))
    torch.cuda.synchronize(dev)
    src, tgt, beta = make_paths(idx, w)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    kk = d["k_per_token"]

    def f_paths(sp, s_=src):
        B.check(B.moe_layer_forward_paths(desc, d["x"], d["w_gate_up"], d["w_down"], s_, tgt,
                                          beta, kk, out, st, ws, sp), "moe_layer_forward_paths")

    def f_diag(sp):
        f_paths(sp, tgt)

    def f_layer(sp):
        B.check(B.moe_layer_forward(desc, d["x"], d["router_w"], d["w_gate_up"], d["w_down"], kk,
                                    out, st, ws, sp), "moe_layer_forward")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    res = {}
    for name, fn in (("paths", f_paths), ("diagonal_paths", f_diag), ("layer", f_layer)):
        with torch.cuda.stream(stream):
            fn(stream.cuda_stream)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            fn(torch.cuda.current_stream().cuda_stream)
        evs = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                if i >= args.warmup:
                    evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        res[name] = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1000.0
        del g
    if B.moe_get_device_status(st) != 0:
        raise RuntimeError("device status after the path runs")
    srcs = src.cpu().numpy()
    kn = kk.cpu().numpy()
    n_exp = int(sum(len(set(srcs[t, :kn[t]].tolist())) for t in range(T)))
    n_paths = int(kn.sum())
    unit = "µs/layer" if wl.phase == "decode" else "tokens/s"
    val = (lambda us: round(us, 2)) if wl.phase == "decode" else \
        (lambda us: round(T / (us * 1e-6), 1))
    return {"metric": "path-composed MoE layer with source-grouped reuse", "unit": unit,
            "higher_is_better": wl.phase != "decode", "n_gpus": world, "dtype": "bf16",
            "data": "synthetic", "steps": args.steps, "warmup": args.warmup,
            "config": {"workload": wl.name, "T": T,
                       "paths": "seeded recipe: consecutive slots share a source"},
            "value": val(res["paths"]),
            "diagonal_paths": val(res["diagonal_paths"]),
            "plain_layer_with_routing": val(res["layer"]),
            "us": {k: round(v, 2) for k, v in res.items()},
            "expansions": n_exp, "paths": n_paths,
            "expansion_flops_saved": 4.0 * H * wl.I_sub * (n_paths - n_exp)}


# The default run: the headline workload first (the line's own value), then
# every other workload, each summarised in the line's "workloads" object.
SWEEP = [("mixtral_decode", None), ("tiny", None), ("qwen_prefill", None),
         ("qwen_decode", 1), ("qwen_decode", 8), ("qwen_decode", 64), ("qwen_decode", 256),
         ("qwen_decode", 1024), ("deepseek_prefill", None)]


def workload_summary(res):
    """The per-workload entry of the sweep: value, roofline, realised routing,
    clocks and the end-to-end number of one run_ours result."""
    keep = ("value", "unit", "higher_is_better", "ms_per_step", "roofline", "roofline_layer",
            "realised", "clocks", "e2e", "breakdown_us", "gpu_launches")
    out = {k: res[k] for k in keep if k in res}
    out["config"] = {k: res["config"][k] for k in ("workload", "T", "l2") if k in res["config"]}
    return out


def profile_calls(args, wl, local):
    """--profile-calls N: N layer calls on one weight copy, nothing timed."""
    import torch
    from aware_moe_expert_gb300 import binding as B
    from aware_moe_expert_gb300.inputs import make_layer_inputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = make_layer_inputs(wl, dev)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    desc.path = args.path
    if args.force_pair:
        desc.debug_flags |= B.DEBUG_FORCE_PAIR
    layer = B.MoeLayer(desc, dev)
    for _ in range(args.profile_calls):
        layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    torch.cuda.synchronize(dev)
    code = layer.device_status()
    return {"mode": "profile-calls", "workload": wl.name, "calls": args.profile_calls,
            "device_status": B.STATUS_NAMES.get(code, code),
            "gb_allocated": round(torch.cuda.max_memory_allocated(dev) / 1e9, 2)}, code


def main():
    args = parse()
    from aware_moe_expert_gb300 import workloads as WL
    sweep = args.workload is None and not args.no_sweep and args.T is None and \
        args.n_experts is None and \
        args.impl == "ours" and not (args.tiered or args.paths or args.profile_calls) and \
        args.router == "linear" and args.fold == 0 and args.k_mode == "exact" and \
        args.k_normal is None and args.path == 0 and not args.force_pair
    wl = WL.ALL[args.workload or "mixtral_decode"]
    if args.T is not None:
        wl = wl.with_T(args.T)
    if args.n_experts is not None:
        wl = wl.with_experts(args.n_experts)
    rank, world, local = dist_info()
    if args.impl == "reference":
        res = run_reference(args, wl, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.profile_calls:
        res, code = profile_calls(args, wl, local)
        print(json.dumps(res), flush=True)
        raise SystemExit(0 if code == 0 else 1)
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.tiered or args.paths:
        res = (run_tiered if args.tiered else run_paths)(args, wl, rank, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res, d = run_ours(args, wl, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_entry(wl, d, args.cpu_budget_s)
    del d
    if sweep:
        import torch
        res["workloads"] = {wl.name: workload_summary(res)}
        launches = res["gpu_launches"]
        for name, T in SWEEP[1:]:
            torch.cuda.empty_cache()
            w2 = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
            r2, d2 = run_ours(args, w2, rank, world, local)
            del d2
            res["workloads"][w2.name] = workload_summary(r2)
            launches += r2["gpu_launches"]
        res["gpu_launches_all_workloads"] = launches
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
