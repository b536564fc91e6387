"""Benchmark of one sparse MoE FFN layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle, timed on host cores

A step is one moe_layer_forward (router GEMM + softmax/top-k, per-expert
capacity selection, dispatch, grouped SwiGLU expert GEMMs, combine, load
statistics) over one synthetic batch resident in HBM. Prints one JSON line.
Under torchrun (N > 1) every rank runs its own replica batch (weak scaling,
no data-path collective); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "mixtral_bf16_gamma1"
METRIC = "MoE-layer tokens/s and grouped-GEMM TFLOP/s (frac. of bf16 peak), 1xB300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms; the
    summary keeps the samples whose timestamps fall inside the timed region."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        # nvidia-smi numbers GPUs its own way; address this one by UUID
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
        except Exception:
            self.gpu = str(cuda_index)
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        deadline = time.time() + 3.0  # let the first samples arrive
        while time.time() < deadline and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except (ValueError, IndexError):
                    continue
        os.remove(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.02 <= r[0] <= self.t1 + 0.02]
        window = "timed region"
        if not inside:
            inside, window = rows, "warm-up and timed region (none inside the timed region)"
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


def count_launches(w, with_stats=True) -> int:
    """Kernels of this library one moe_layer_forward launches."""
    n = 1 + 1 + 1 + 1 + 2 + 1          # logits, route, select, dispatch, 2 GEMMs, combine
    if w.f_shared:
        n += 1 + 2                      # shared offsets, 2 GEMMs
    if with_stats:
        n += 2 if w.T > 0 else 1
    return n


def ffn_flops(w, P: int) -> float:
    return 6.0 * w.d * w.f * P + (6.0 * w.d * w.f_shared * w.T if w.f_shared else 0.0)


def stage_bytes(w, P: int):
    sx = 2 if w.dtype == "bf16" else 4
    kc = w.N if w.mode == W.EXPERT_CHOICE else w.k + w.m
    return {
        "route": w.T * w.d * sx + w.d * w.N * sx + w.T * w.N * 4 * 2 + w.T * kc * 8,
        "dispatch": w.T * w.d * sx + P * w.d * sx + 16 * P,
        "combine": P * w.d * sx + w.T * w.d * sx + 8 * P + (w.T * w.d * sx if w.f_shared else 0),
    }


def cpu_oracle_sample(w, n_tokens: int):
    """The oracle, as it stands, on a bounded sample: full-batch routing (the
    capacity couples all tokens) plus the expert FFN of n_tokens tokens."""
    import oracle as O
    inp = W.make_inputs(w)
    f = lambda t: None if t is None else t.float().numpy()  # noqa: E731
    x, Wr, b = f(inp["x"]), f(inp["W_r"]), f(inp["bias"])
    W1, W3, W2 = f(inp["W1"]), f(inp["W3"]), f(inp["W2"])
    Ws = [f(inp.get(k)) for k in ("Ws1", "Ws3", "Ws2")]
    rng = np.random.default_rng(0)
    tokens = np.sort(rng.choice(w.T, size=min(n_tokens, w.T), replace=False))
    t0 = time.perf_counter()
    O.layer_forward(x, Wr, b, W1, W3, W2, mode=w.mode, k=w.k, gamma=w.gamma, m=w.m,
                    group_size=w.group_size, renorm=w.renorm, dtype=w.dtype, Ws1=Ws[0],
                    Ws3=Ws[1], Ws2=Ws[2], tokens=tokens)
    dt = time.perf_counter() - t0
    return len(tokens), dt


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed on the host cores."""
    if rank != 0:
        return
    w = W.ALL[args.workload]
    n_tok = args.cpu_sample_tokens
    for _ in range(args.warmup):
        cpu_oracle_sample(w, n_tok)
    times = []
    for _ in range(args.steps):
        n, dt = cpu_oracle_sample(w, n_tok)
        times.append(dt)
    tps = n / statistics.mean(times)
    cores = os.cpu_count()  # OpenBLAS runs the fp64 matmuls on every core
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(), "sample_tokens": n},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"full-batch routing + expert FFN of {n} of {w.T} tokens"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.ALL[args.workload]
    dist = world > 1
    if dist:
        import torch.distributed as td

    inp = W.make_inputs(w.replace(seed=w.seed + rank) if args.distinct_batches else w)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    cfg = M.config_from_workload(w)
    sz = M.sizes(cfg)
    ws = torch.zeros(sz.workspace, dtype=torch.uint8, device=dev)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((w.T, w.d), dtype=dt, device=dev)
    stats = torch.zeros(M.MOE_STATS_LEN, dtype=torch.float64, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        M.moe_layer_forward(cfg, d["x"], d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"],
                            d.get("Ws1"), d.get("Ws3"), d.get("Ws2"), y, ws, stats=stats,
                            stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if M.moe_get_device_status(ws) != M.MOE_OK:
        raise RuntimeError("device status error after warm-up")
    st = stats.cpu().numpy()
    P = int(st[0])

    # ---- timed region: K steps, L2 flushed between steps (outside the events) ----
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    if dist:
        td.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.nvtx.range_push("moe_timed_steps")
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    if dist:
        td.barrier()
    ms = [a.elapsed_time(b) for a, b in evs]
    clk = clocks.stop() if clocks else None
    total_ms = sum(ms)
    if dist:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        td.all_reduce(t, op=td.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = world * w.T * args.steps / (total_ms / 1e3)

    # ---- the expert GEMMs on their own (the dominant kernel), same rows ----
    v = M.moe_workspace_views(cfg, ws)
    offs = M.view_tensor(v.expert_offsets, (w.N + 1,), torch.int32)
    xp = M.view_tensor(v.xp, (int(sz.rows_max), w.d), dt)
    op = M.view_tensor(v.op, (int(sz.rows_max), w.d), dt)
    ffn_ws = torch.zeros(M.ffn_workspace_size(int(sz.rows_max), w.f, w.dtype), dtype=torch.uint8,
                         device=dev)
    kreps = max(3, args.steps)
    for _ in range(2):
        M.moe_expert_ffn(cfg, xp, offs, w.N, int(sz.rows_max), w.f, d["W1"], d["W3"], d["W2"], op,
                         ffn_ws, stream=stream)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(kreps)]
    for a, b in fev:
        flush.zero_()
        a.record(stream)
        M.moe_expert_ffn(cfg, xp, offs, w.N, int(sz.rows_max), w.f, d["W1"], d["W3"], d["W2"], op,
                         ffn_ws, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    ffn_ms = statistics.mean(a.elapsed_time(b) for a, b in fev)
    routed_flops = 6.0 * w.d * w.f * P
    ffn_tflops = routed_flops / (ffn_ms * 1e-3) / 1e12

    # ---- HBM-bound stages on their own (split entry points, same buffers) ----
    kc = sz.kc
    scores = M.view_tensor(v.scores, (w.T, w.N), torch.float32)
    cand_idx = M.view_tensor(v.cand_idx, (w.T, kc), torch.int32)
    cand_gate = M.view_tensor(v.cand_gate, (w.T, kc), torch.float32)
    slot = M.view_tensor(v.slot, (w.T, kc), torch.int32)
    keep = M.view_tensor(v.keep, (w.T, kc), torch.uint8)
    demand = M.view_tensor(v.demand, (w.N,), torch.int32)
    kept = M.view_tensor(v.kept, (w.N,), torch.int32)
    row_token = M.view_tensor(v.row_token, (int(sz.rows_max),), torch.int32)
    row_gate = M.view_tensor(v.row_gate, (int(sz.rows_max),), torch.float32)
    tok_rows = M.view_tensor(v.tok_rows, (w.T, kc), torch.int32)
    logits = M.view_tensor(v.logits, (w.T, w.N), torch.float32)
    ec = w.mode == W.EXPERT_CHOICE
    rws = torch.zeros(M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    stages = {
        "route": lambda: M.moe_route(cfg, d["x"], d["W_r"], d["bias"], logits, scores,
                                     None if ec else cand_idx, cand_gate, rws, stream=stream),
        "select": lambda: M.moe_capacity_drop(cfg, None if ec else cand_idx, cand_gate, slot, keep,
                                              demand, kept, stream=stream),
        "dispatch": lambda: M.moe_dispatch(cfg, d["x"], None if ec else cand_idx, cand_gate, slot,
                                           kept, offs, row_token, row_gate, tok_rows, xp,
                                           stream=stream),
        "combine": lambda: M.moe_combine(cfg, op, row_gate, tok_rows,
                                         M.view_tensor(v.shared_out, (w.T, w.d), dt)
                                         if w.f_shared else None, y, stream=stream),
    }
    stage_ms = {}
    for name, fn in stages.items():
        fn()
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(kreps)]
        for a, b in sev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        stage_ms[name] = statistics.mean(a.elapsed_time(b) for a, b in sev)

    # ---- end to end through host buffers: H2D x, layer, D2H y every step ----
    x_host = inp["x"].pin_memory()
    y_host = torch.empty((w.T, w.d), dtype=dt).pin_memory()
    x_dev = torch.empty_like(d["x"])

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        M.moe_layer_forward(cfg, x_dev, d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"],
                            d.get("Ws1"), d.get("Ws3"), d.get("Ws2"), y, ws, stats=stats,
                            stream=stream)
        y_host.copy_(y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if dist:
        t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
        td.all_reduce(t, op=td.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * w.T * args.steps / (e2e_ms / 1e3)
    sx = 2 if w.dtype == "bf16" else 4

    if M.moe_get_device_status(ws) != M.MOE_OK:
        raise RuntimeError("device status error in the timed region")
    if rank != 0:
        return

    peaks, peak_src = load_peaks()
    peak_tf = float(peaks["bf16_tflops"])
    sbytes = stage_bytes(w, P)
    hbm = float(peaks["hbm_gbs"])
    kernels = {}
    for name in ("route", "dispatch", "combine"):
        gbs = sbytes[name] / (stage_ms[name] * 1e-3) / 1e9
        kernels[name] = {"ms": stage_ms[name], "bytes": sbytes[name], "GB/s": gbs,
                         "frac_hbm": gbs / hbm}
    kernels["select"] = {"ms": stage_ms["select"]}
    kernels["expert_ffn"] = {"ms": ffn_ms, "flops": routed_flops, "TFLOP/s": ffn_tflops,
                             "frac_bf16": ffn_tflops / peak_tf}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n, t_cpu = cpu_oracle_sample(w, args.cpu_sample_tokens)
        cpu = {"value": n / t_cpu, "unit": "tokens/s", "cores": os.cpu_count(),
               "kind": "oracle",
               "sample": f"full-batch routing + expert FFN of {n} of {w.T} tokens ({t_cpu:.1f} s)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.describe(), "T": w.T, "d": w.d, "N": w.N, "f": w.f, "k": w.k,
                   "mode": w.mode, "gamma": None if math.isinf(w.gamma) else w.gamma,
                   "kept_pairs": P, "l2": "flushed (256 MiB write) before every timed step",
                   "parallelism": f"replicas x{world}"},
        "tflops": ffn_flops(w, P) * args.steps * world / (total_ms / 1e3) / 1e12,
        "roofline": {"kernel": "grouped_gemm_tc (GEMM1+SwiGLU and GEMM2, one launch each)",
                     "bound": "tensor", "achieved": ffn_tflops, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": ffn_tflops / peak_tf, "traffic": None,
                     "peak_source": f"{peak_src} bf16 burst"},
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * sx,
                "d2h_bytes_per_step": w.T * w.d * sx},
        "gpu_launches": count_launches(w) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "stats": {"max_over_mean": float(st[4]), "drop_fraction": float(st[5]),
                  "balance_times_N": float(st[7])},
    }
    print(json.dumps(line), flush=True)


def run_stage(args):
    """--kernel STAGE: loop one stage of the layer on the workload (T
    overridable with --T) and print its device time and algorithmic GB/s.
    Holds only the routing-side tensors on the device, so a single kernel can
    be profiled with ncu on inputs larger than L2."""
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = W.ALL[args.workload]
    if args.T:
        w = w.replace(T=args.T)
    inp = W.make_inputs(w, with_experts=False)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    cfg = M.config_from_workload(w)
    sz = M.sizes(cfg)
    R, kc = int(sz.rows_max), sz.kc
    ec = w.mode == W.EXPERT_CHOICE
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    f32, i32 = torch.float32, torch.int32
    logits = torch.empty((w.T, w.N), dtype=f32, device=dev)
    scores = torch.empty((w.T, w.N), dtype=f32, device=dev)
    cand_idx = torch.empty((w.T, kc), dtype=i32, device=dev)
    cand_gate = torch.empty((w.T, kc), dtype=f32, device=dev)
    slot = torch.empty((w.T, kc), dtype=i32, device=dev)
    keep = torch.empty((w.T, kc), dtype=torch.uint8, device=dev)
    demand = torch.empty((w.N,), dtype=i32, device=dev)
    kept = torch.empty((w.N,), dtype=i32, device=dev)
    offs = torch.empty((w.N + 1,), dtype=i32, device=dev)
    row_token = torch.empty((R,), dtype=i32, device=dev)
    row_gate = torch.empty((R,), dtype=f32, device=dev)
    tok_rows = torch.empty((w.T, kc), dtype=i32, device=dev)
    xp = torch.empty((R, w.d), dtype=dt, device=dev)
    op = torch.zeros((R, w.d), dtype=dt, device=dev)
    y = torch.empty((w.T, w.d), dtype=dt, device=dev)
    rws = torch.zeros(M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    ci = None if ec else cand_idx
    fns = {
        "route": lambda: M.moe_route(cfg, d["x"], d["W_r"], d["bias"], logits, scores, ci,
                                     cand_gate, rws),
        "select": lambda: M.moe_capacity_drop(cfg, ci, cand_gate, slot, keep, demand, kept),
        "dispatch": lambda: M.moe_dispatch(cfg, d["x"], ci, cand_gate, slot, kept, offs,
                                           row_token, row_gate, tok_rows, xp),
        "combine": lambda: M.moe_combine(cfg, op, row_gate, tok_rows, None, y),
    }
    for name in ("route", "select", "dispatch"):
        fns[name]()
    torch.cuda.synchronize()
    P = int(offs[-1].item())
    fn = fns[args.kernel]
    for _ in range(args.warmup):
        flush.zero_()
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.nvtx.range_push("moe_stage")
    for a, b in evs:
        flush.zero_()
        a.record()
        fn()
        b.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = stage_bytes(w, P).get(args.kernel)
    peaks, src = load_peaks()
    out = {"kernel": args.kernel, "workload": w.describe(), "kept_pairs": P, "ms": ms}
    if nbytes:
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.update({"bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / float(peaks["hbm_gbs"]),
                    "peak_source": src})
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.ALL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=256)
    ap.add_argument("--distinct-batches", action="store_true",
                    help="each rank draws its own x (seed + rank)")
    ap.add_argument("--kernel", choices=["route", "select", "dispatch", "combine"],
                    help="time one stage alone instead of the layer")
    ap.add_argument("--T", type=int, default=0, help="token count override for --kernel")
    args = ap.parse_args()
    if args.kernel:
        run_stage(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as td
        torch.cuda.set_device(local_rank)
        td.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as td
            td.destroy_process_group()


if __name__ == "__main__":
    main()
