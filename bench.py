"""Benchmark of one sparse MoE FFN layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle, timed on host cores
    python bench.py --vs-cublas --steps 10   # plain grouped GEMM beside cuBLAS bmm

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


def layer_call(M, cfg, w, d, x, y, ws, stats=None, stream=None):
    """One moe_layer_forward (moe_layer_forward_e4m3 for FP8 routed experts)."""
    if w.weights == "e4m3":
        ex = M.e4m3_experts(d["W1q"], d["W3q"], d["W2q"], d["W1s"], d["W3s"], d["W2s"])
        M.moe_layer_forward_e4m3(cfg, x, d["W_r"], d["bias"], ex, d.get("Ws1"), d.get("Ws3"),
                                 d.get("Ws2"), y, ws, stats=stats, stream=stream)
    else:
        M.moe_layer_forward(cfg, x, d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"], d.get("Ws1"),
                            d.get("Ws3"), d.get("Ws2"), y, ws, stats=stats, stream=stream)


def routed_weight_bytes(w, kept) -> int:
    """Bytes of the routed experts a step reads: the weights (and column
    scales) of every expert that kept at least one row."""
    per = 3 * w.d * w.f * (1 if w.weights == "e4m3" else (2 if w.dtype == "bf16" else 4))
    if w.weights == "e4m3":
        per += 4 * (2 * w.f + w.d)
    return per * int((np.asarray(kept) > 0).sum())


def ffn_flops(w, P: int) -> float:
    return 6.0 * w.d * w.f * P + (6.0 * w.d * w.f_shared * w.T if w.f_shared else 0.0)


def stage_bytes(w, P: int, fused_gather: bool = False):
    sx = 2 if w.dtype == "bf16" else 4
    kc = w.N if w.mode == W.EXPERT_CHOICE else w.k + w.m
    return {
        "route": w.T * w.d * sx + w.d * w.N * sx + w.T * w.N * 4 * 2 + w.T * kc * 8,
        # with the gather fused into GEMM1 dispatch moves only the row tables
        "dispatch": (0 if fused_gather else w.T * w.d * sx + P * w.d * sx) + 16 * P,
        "combine": P * w.d * sx + w.T * w.d * sx + 8 * P + (w.T * w.d * sx if w.f_shared else 0),
    }


def _blas_threads() -> int:
    """Threads the oracle's fp64 BLAS calls actually run on."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


class OracleSampler:
    """The oracle, as it stands, on bounded samples of one workload: the
    routing of the whole batch (capacity and expert choice couple all tokens)
    plus the expert FFN of a fixed random subset of tokens. The subset size is
    calibrated once so that one sample takes about ``target_s`` seconds."""

    def __init__(self, w):
        import oracle as O
        self.O = O
        self.w = w
        inp = W.make_inputs(w)
        f = lambda t: None if t is None else t.float().numpy()  # noqa: E731
        if w.weights == "e4m3":  # the experts the library multiplies
            Wx = [O.dequantize_e4m3(inp[n + "q"].numpy(), inp[n + "s"].numpy(), kmajor=True)
                  for n in ("W1", "W3", "W2")]
        else:
            Wx = [f(inp[n]) for n in ("W1", "W3", "W2")]
        self.args = (f(inp["x"]), f(inp["W_r"]), f(inp["bias"]), *Wx)
        self.shared = [f(inp.get(k)) for k in ("Ws1", "Ws3", "Ws2")]
        self.n_tokens = None

    def run(self, n_tokens: int):
        w = self.w
        rng = np.random.default_rng(0)
        tokens = np.sort(rng.choice(w.T, size=min(n_tokens, w.T), replace=False))
        t0 = time.perf_counter()
        self.O.layer_forward(*self.args, mode=w.mode, k=w.k, gamma=w.gamma, m=w.m,
                             group_size=w.group_size, renorm=w.renorm, dtype=w.dtype,
                             Ws1=self.shared[0], Ws3=self.shared[1], Ws2=self.shared[2],
                             tokens=tokens, act_e4m3=w.weights == "e4m3")
        return len(tokens), time.perf_counter() - t0

    def calibrate(self, target_s: float) -> int:
        """Pick the token count whose sample takes about target_s seconds."""
        self.run(min(16, self.w.T))  # first call: thread pools and page faults
        n0, t0 = self.run(min(64, self.w.T))
        n1, t1 = self.run(min(256, self.w.T))
        per_tok = max((t1 - t0) / max(n1 - n0, 1), 1e-6)
        fixed = max(t0 - per_tok * n0, 0.0)  # full-batch routing
        n = int((target_s - fixed) / per_tok)
        self.n_tokens = max(1, min(self.w.T, n))
        return self.n_tokens

    def describe(self, n: int, dt: float) -> str:
        return (f"full-batch routing of {self.w.T} tokens + expert FFN of {n} of them "
                f"(one sample, {dt:.1f} s)")


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed on the host cores."""
    if rank != 0:
        return
    w = W.ALL[args.workload]
    smp = OracleSampler(w)
    # whole run (warm-up + timed) bounded to about args.reference_budget_s
    per_step = min(20.0, max(1.0, args.reference_budget_s / max(1, args.steps + args.warmup)))
    n_tok = smp.calibrate(per_step)
    for _ in range(args.warmup):
        smp.run(n_tok)
    times = []
    for _ in range(args.steps):
        n, dt = smp.run(n_tok)
        times.append(dt)
    tps = n / statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe(), "sample_tokens": n},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": _blas_threads(),
                         "kind": "oracle",
                         "sample": smp.describe(n, statistics.mean(times)) + " per step"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(ms: float, dev) -> float:
    """The slowest rank's time: every rank calls this with its own; without
    an initialised process group it returns `ms` unchanged."""
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()):
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: int, steps: int, ms: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes
    `units_per_rank` units per step, and the job takes the slowest rank's
    time `ms` for `steps` steps."""
    return world * units_per_rank * steps / (ms / 1e3)


def gemm_traffic(w):
    """DRAM bytes per launch of the grouped GEMM pair on this workload from
    the committed ncu capture, or None when the kernel source differs from
    the one captured (the counters no longer describe it)."""
    import hashlib
    src = os.path.join(ROOT, "routing_capacity_drop_router_b300", "csrc", "ffn_tcgen05.cu")
    with open(src, "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()[:16]
    rec = GEMM_TRAFFIC.get(w.name)
    if rec is None or rec["kernel_sha"] != sha:
        return None
    return rec["bytes_per_launch_pair"]


# dram__bytes_read.sum + dram__bytes_write.sum of expert_gemm1_swiglu +
# expert_gemm2 from one ncu capture per workload,
# keyed by the sha256 prefix of the kernel source it was taken on.
GEMM_TRAFFIC = {
    # the CTA-pair grouped GEMM on the Mixtral-shaped layer at gamma 1: GEMM1+SwiGLU
    # 2.009582 GB read + 0.140430 GB written, GEMM2 1.181581 GB + 0.039514 GB
    "mixtral_bf16_gamma1": {"kernel_sha": "9ea6ad912332f037",
                            "bytes_per_launch_pair": 2.009582e9 + 0.140430e9 +
                            1.181581e9 + 0.039514e9},
}


def device_inputs(w, dev, rank=0, distinct=False):
    """The workload's seeded inputs on the device (e4m3 experts: only the
    bytes and scales), plus the host copy of x for the end-to-end leg."""
    inp = W.make_inputs(w.replace(seed=w.seed + rank) if distinct else w)
    if w.weights == "e4m3":  # the routed experts live on the device in e4m3 only
        inp = {k: v for k, v in inp.items() if k not in ("W1", "W3", "W2")}
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    return d, inp["x"]


def roofline_of(w, P, kept_h, g1, g2, peaks, peak_src):
    """Roofline of the expert GEMMs (GEMM1+SwiGLU and GEMM2 event times, ms):
    tensor-bound at the kept pairs' 6*d*f flops, or HBM-bound on the bytes of
    the experts hit plus the rows in and out when the flops per byte fall
    below the machine balance (decode batches)."""
    peak_tf = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    routed_flops = 6.0 * w.d * w.f * P
    sx = 2 if w.dtype == "bf16" else 4
    gemm_bytes = routed_weight_bytes(w, kept_h) + 2 * P * (w.d + w.f) * sx
    sec = (g1 + g2) * 1e-3
    tflops = routed_flops / sec / 1e12
    gbs = gemm_bytes / sec / 1e9
    ridge = peak_tf * 1e12 / (hbm * 1e9)
    if routed_flops / gemm_bytes < ridge:
        return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "algorithmic_bytes": gemm_bytes, "peak_source": f"{peak_src} HBM copy",
                "tflops": tflops}
    return {"bound": "tensor", "achieved": tflops, "peak": peak_tf, "unit": "TFLOP/s",
            "frac": tflops / peak_tf, "peak_source": f"{peak_src} bf16 burst",
            "frac_of_sustained": tflops / float(peaks.get("bf16_tflops_sustained", peak_tf)),
            "flops_per_byte": routed_flops / gemm_bytes, "machine_balance": ridge,
            "hbm_view": {"achieved": gbs, "unit": "GB/s", "frac": gbs / hbm,
                         "algorithmic_bytes": gemm_bytes}}


def measure_layer(M, w, d, args, dev, world, rank, fuse_gather=False):
    """Warm-up, then args.steps timed moe_layer_forward steps (events only at
    the step boundaries and around the expert GEMMs, clocks sampled inside
    the timed region, max over ranks), then a pass with an event at every
    kernel boundary for the per-stage times. Returns the measurements and the
    state the end-to-end leg reuses."""
    import torch.distributed as td
    dist = world > 1
    cfg = M.config_from_workload(w, fuse_gather=fuse_gather)
    wsz = M.workspace_size_e4m3(cfg) if w.weights == "e4m3" else M.sizes(cfg).workspace
    ws = torch.zeros(wsz, dtype=torch.uint8, device=dev)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((w.T, w.d), dtype=dt, device=dev)
    stats = torch.zeros(M.MOE_STATS_LEN, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    stages = M.moe_layer_stages(cfg)
    weight_bytes = sum(t.numel() * t.element_size() for k, t in d.items()
                       if t is not None and k in ("W1", "W3", "W2", "Ws1", "Ws3", "Ws2",
                                                  "W1q", "W3q", "W2q"))
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    # Between steps the L2 is not flushed when every step streams expert
    # weights far larger than the L2 through it (the next step's activations
    # start cold); smaller workloads flush explicitly.
    flush = None
    if weight_bytes < 4 * l2_bytes:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def step():
        layer_call(M, cfg, w, d, d["x"], y, ws, stats=stats, stream=stream)

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    if M.moe_get_device_status(ws) != M.MOE_OK:
        raise RuntimeError(f"{w.name}: device status error after warm-up")
    st = stats.cpu().numpy()
    P = int(st[0])
    vw = M.moe_workspace_views(cfg, ws)
    kept_h = M.view_tensor(vw.kept, (w.N,), torch.int32, dev).cpu().numpy()
    coverage = M.view_tensor(vw.coverage, (w.T,), torch.int32, dev).cpu().numpy()

    # ---- timed region: K layer steps. The library records events on the
    # launching stream at the step's start and end and around the expert GEMMs
    # (the dominant kernels); other kernel boundaries get no event, so their
    # launches overlap (programmatic dependent launch) as in normal use ----
    g1_i = stages.index("expert_gemm1_swiglu")
    timed_at = {0, g1_i, g1_i + 1, g1_i + 2, len(stages)}

    def new_row(marks):
        return [torch.cuda.Event(enable_timing=True) if i in marks else None
                for i in range(len(stages) + 1)]

    evs = [new_row(timed_at) for _ in range(args.steps)]
    for row in evs:  # give every event its CUDA handle before the timed region
        for e in row:
            if e is not None:
                e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    if dist:
        td.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    torch.cuda.nvtx.range_push("moe_timed_steps")
    for row in evs:
        if flush is not None:
            flush.zero_()
        M.moe_set_trace_events(row)
        step()
    M.moe_set_trace_events(None)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    if dist:
        td.barrier()
    clk = clocks.stop() if clocks else None
    step_ms = [row[0].elapsed_time(row[-1]) for row in evs]
    total_ms = sum(step_ms) if flush is not None else evs[0][0].elapsed_time(evs[-1][-1])
    g1_ms = statistics.mean(row[g1_i].elapsed_time(row[g1_i + 1]) for row in evs)
    g2_ms = statistics.mean(row[g1_i + 1].elapsed_time(row[g1_i + 2]) for row in evs)
    # the stages around the expert GEMMs as they overlap in the timed steps
    pre_ms = statistics.mean(row[0].elapsed_time(row[g1_i]) for row in evs)
    post_ms = statistics.mean(row[g1_i + 2].elapsed_time(row[-1]) for row in evs)
    total_ms = max_over_ranks(total_ms, dev)

    # ---- per-kernel breakdown: a few more steps with an event at every
    # kernel boundary (this serialises the launches) ----
    n_tr = max(3, min(args.steps, 20))
    tr = [new_row(set(range(len(stages) + 1))) for _ in range(n_tr)]
    for row in tr:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for row in tr:
        if flush is not None:
            flush.zero_()
        M.moe_set_trace_events(row)
        step()
    M.moe_set_trace_events(None)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(row[i].elapsed_time(row[i + 1]) for row in tr)
                for i, name in enumerate(stages)}
    if M.moe_get_device_status(ws) != M.MOE_OK:
        raise RuntimeError(f"{w.name}: device status error in the timed region")
    return dict(cfg=cfg, ws=ws, y=y, stats=stats, st=st, P=P, kept_h=kept_h, coverage=coverage,
                stages=stages, stream=stream, flush=flush, weight_bytes=weight_bytes,
                l2_bytes=l2_bytes, total_ms=total_ms, g1=g1_ms, g2=g2_ms, pre=pre_ms,
                post=post_ms, stage_ms=stage_ms, clocks=clk)


def kernel_table(w, r, peaks, fused_gather=False):
    """Per-kernel figures: the HBM-bound stages' algorithmic GB/s, the
    selection's time, the expert GEMMs' flops rate and the stage times."""
    hbm = float(peaks["hbm_gbs"])
    P, stage_ms = r["P"], r["stage_ms"]
    sbytes = stage_bytes(w, P, fused_gather=fused_gather)
    kernels = {}
    route_ms = sum(stage_ms.get(n, 0.0) for n in ("router", "router_logits", "route_tokens"))
    for name, ms in (("route", route_ms), ("dispatch", stage_ms["dispatch"]),
                     ("combine", stage_ms["combine"])):
        gbs = sbytes[name] / (ms * 1e-3) / 1e9
        kernels[name] = {"ms": ms, "bytes": sbytes[name], "GB/s": gbs, "frac_hbm": gbs / hbm}
    kernels["select"] = {"ms": stage_ms["select"]}
    g1, g2 = r["g1"], r["g2"]
    kernels["expert_gemm1_swiglu"] = {"ms": g1, "flops": 4.0 * w.d * w.f * P,
                                      "TFLOP/s": 4.0 * w.d * w.f * P / (g1 * 1e-3) / 1e12}
    kernels["expert_gemm2"] = {"ms": g2, "flops": 2.0 * w.d * w.f * P,
                               "TFLOP/s": 2.0 * w.d * w.f * P / (g2 * 1e-3) / 1e12}
    if w.f_shared and "shared_gemm1_swiglu" in stage_ms:
        sg = stage_ms["shared_gemm1_swiglu"] + stage_ms["shared_gemm2"]
        kernels["shared_expert"] = {"ms": sg, "flops": 6.0 * w.d * w.f_shared * w.T,
                                    "TFLOP/s": 6.0 * w.d * w.f_shared * w.T / (sg * 1e-3) / 1e12}
    kernels["stage_ms_serialised"] = stage_ms
    kernels["timed_steps_ms"] = {"before_expert_gemms": r["pre"], "expert_gemms": g1 + g2,
                                 "after_expert_gemms": r["post"]}
    return kernels


def coverage_summary(cov):
    """How many experts took each token (expert choice: some tokens are taken
    by several experts, some by none)."""
    cov = np.asarray(cov)
    if cov.size == 0:
        return None
    return {"min": int(cov.min()), "max": int(cov.max()), "mean": float(cov.mean()),
            "zero_coverage_tokens": int((cov == 0).sum()),
            "histogram": {str(int(v)): int(c) for v, c in zip(*np.unique(cov, return_counts=True))}}


# Further workloads measured after the headline one, each in the same way and
# reported in the line's "configs" object: the Mixtral-shaped layer without a
# capacity limit and at capacity factor 1.5, the fine-grained layer with its
# shared expert, the expert-choice layer and the decode batch.
EXTRA_CONFIGS = ("mixtral_bf16", "mixtral_bf16_gamma1.5", "finegrained_bf16",
                 "expert_choice_bf16", "decode_bf16", "decode_e4m3")


def e4m3_from_bf16(d):
    """The e4m3 experts of a workload whose bf16 draws are already on the
    device (the recipe's per-column quantization, done on the GPU here, stored
    K-major); the bf16 routed experts are dropped."""
    out = {k: v for k, v in d.items() if k not in ("W1", "W3", "W2")}
    for name in ("W1", "W3", "W2"):
        q, sc = W.quantize_e4m3(d[name])
        out[name + "q"], out[name + "s"] = q.transpose(-1, -2).contiguous(), sc
    return out


def config_entry(w, r, args, world, peaks, peak_src):
    """One workload's entry of the "configs" object."""
    roof = roofline_of(w, r["P"], r["kept_h"], r["g1"], r["g2"], peaks, peak_src)
    kern = kernel_table(w, r, peaks)
    st = r["st"]
    out = {
        "workload": w.describe(), "steps": args.steps, "warmup": args.warmup,
        "tokens_per_s": job_rate(world, w.T, args.steps, r["total_ms"]),
        "ms_per_step": r["total_ms"] / args.steps, "kept_pairs": r["P"],
        "gemm1_us": 1e3 * r["g1"], "gemm2_us": 1e3 * r["g2"],
        "roofline": roof,
        "hbm_stages": {k: {"GB/s": kern[k]["GB/s"], "frac_hbm": kern[k]["frac_hbm"],
                           "ms": kern[k]["ms"]} for k in ("route", "dispatch", "combine")},
        "select_ms": kern["select"]["ms"],
        "timed_steps_ms": kern["timed_steps_ms"],
        "stats": {"max_over_mean": float(st[4]), "drop_fraction": float(st[5]),
                  "balance_times_N": float(st[7])},
        "clocks": r["clocks"],
        "l2": "flushed before every timed step" if r["flush"] is not None else "not flushed",
    }
    if "shared_expert" in kern:
        out["shared_expert_us"] = 1e3 * kern["shared_expert"]["ms"]
    if w.mode == W.EXPERT_CHOICE:
        out["coverage"] = coverage_summary(r["coverage"])
    return out


def run_ours(args, rank, world, local_rank):
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.ALL[args.workload]
    dist = world > 1
    if dist:
        import torch.distributed as td

    d, x_cpu = device_inputs(w, dev, rank, args.distinct_batches)
    fused = args.gather == "fused"
    r = measure_layer(M, w, d, args, dev, world, rank, fuse_gather=fused)
    cfg, ws, y, stats, stream = r["cfg"], r["ws"], r["y"], r["stats"], r["stream"]
    total_ms, st, P = r["total_ms"], r["st"], r["P"]
    ms_per_step = total_ms / args.steps
    value = job_rate(world, w.T, args.steps, total_ms)
    dt = y.dtype

    # ---- end to end through host buffers: every step copies its x from
    # pinned host memory, runs the layer and copies y back to pinned host
    # memory. Three streams pipeline the steps as a server would: step i+1's
    # upload and step i-1's download overlap step i's layer (double-buffered
    # device x and y; events order the reuse of each buffer) ----
    x_host = x_cpu.pin_memory()
    y_host = [torch.empty((w.T, w.d), dtype=dt).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(d["x"]) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    s_up = torch.cuda.Stream(dev)
    s_down = torch.cuda.Stream(dev)
    up_done = [torch.cuda.Event() for _ in range(2)]
    layer_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(layer_done[b])  # step i-2 has read x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                up_done[b].record(s_up)
            stream.wait_event(up_done[b])
            if i >= 2:
                stream.wait_event(down_done[b])  # step i-2's y_dev[b] is on the host
            layer_call(M, cfg, w, d, x_dev[b], y_dev[b], ws, stats=stats, stream=stream)
            layer_done[b].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(layer_done[b])
                y_host[b].copy_(y_dev[b], non_blocking=True)
                down_done[b].record(s_down)
        # the region ends when the last download has landed
        for ev in down_done:
            stream.wait_event(ev)

    e2e_steps(2)
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    if not torch.equal(y_host[(args.steps - 1) & 1], y.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    e2e_value = job_rate(world, w.T, args.steps, e2e_ms)
    sx = 2 if w.dtype == "bf16" else 4
    if M.moe_get_device_status(ws) != M.MOE_OK:
        raise RuntimeError("device status error in the end-to-end steps")

    peaks, peak_src = load_peaks()
    fused_stage = fused and w.dtype == "bf16" and w.weights == "same"
    roof = roofline_of(w, P, r["kept_h"], r["g1"], r["g2"], peaks, peak_src)
    kernels = kernel_table(w, r, peaks, fused_gather=fused_stage)

    # ---- the other workloads, each measured the same way (one GPU only:
    # the replica runs under torchrun time the headline workload alone) ----
    configs = None
    if world == 1 and not args.no_configs:
        del x_host, y_host, x_dev, y_dev
        configs = {}
        cache = {w.name: d} if w.T == W.MIXTRAL_BF16.T and w.d == W.MIXTRAL_BF16.d and \
            w.N == W.MIXTRAL_BF16.N and w.f == W.MIXTRAL_BF16.f and w.weights == "same" and \
            w.seed == W.MIXTRAL_BF16.seed and not args.distinct_batches else {}
        for name in EXTRA_CONFIGS:
            if name == w.name:
                continue
            wx = W.ALL[name]
            same_draws = [k for k, v in cache.items()
                          if (W.ALL[k].T, W.ALL[k].d, W.ALL[k].N, W.ALL[k].f, W.ALL[k].f_shared,
                              W.ALL[k].zipf_s, W.ALL[k].dtype, W.ALL[k].weights) ==
                          (wx.T, wx.d, wx.N, wx.f, wx.f_shared, wx.zipf_s, wx.dtype, wx.weights)]
            if same_draws:  # the same draws (only the routing mode differs)
                dx = cache[same_draws[0]]
            elif wx.weights == "e4m3" and \
                    any(W.ALL[k] == wx.replace(name=k, weights="same") for k in cache):
                # e4m3 experts quantized from the bf16 draws already on the device
                k0 = next(k for k in cache if W.ALL[k] == wx.replace(name=k, weights="same"))
                dx = e4m3_from_bf16(cache.pop(k0))
                torch.cuda.empty_cache()
                cache[name] = dx
            else:
                cache.clear()
                torch.cuda.empty_cache()
                dx, _ = device_inputs(wx, dev)
                cache[name] = dx
            rx = measure_layer(M, wx, dx, args, dev, world, rank)
            configs[name] = config_entry(wx, rx, args, world, peaks, peak_src)
            del rx
        cache.clear()
        torch.cuda.empty_cache()

    if rank != 0:
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(w)
        n_tok = smp.calibrate(args.cpu_sample_s)
        n, t_cpu = smp.run(n_tok)
        if t_cpu < 0.5 * args.cpu_sample_s and n < w.T:  # calibration undershot: one larger sample
            n, t_cpu = smp.run(min(w.T, int(n * args.cpu_sample_s / max(t_cpu, 1e-3))))
        cpu = {"value": n / t_cpu, "unit": "tokens/s", "cores": _blas_threads(),
               "kind": "oracle", "sample": smp.describe(n, t_cpu)}

    flush, weight_bytes, l2_bytes = r["flush"], r["weight_bytes"], r["l2_bytes"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.describe(), "T": w.T, "d": w.d, "N": w.N, "f": w.f, "k": w.k,
                   "mode": w.mode, "gamma": None if math.isinf(w.gamma) else w.gamma,
                   "kept_pairs": P,
                   "gather": ("fused into expert GEMM1 (MOE_FUSE_GATHER)"
                              if fused_stage else "dispatch copies the token rows"),
                   "l2": ("flushed (256 MiB write) before every timed step" if flush is not None
                          else f"not flushed: inputs larger than L2 ({weight_bytes / 1e9:.2f} GB "
                               f"of expert weights stream through the {l2_bytes / 2**20:.0f} MiB "
                               "L2 every step)"),
                   "parallelism": f"replicas x{world}"},
        "tflops": ffn_flops(w, P) * args.steps * world / (total_ms / 1e3) / 1e12,
        "roofline": dict({"kernel": ("grouped_gemm_w8_kernel" if w.weights == "e4m3" else
                                     "grouped_gemm_tc_kernel") +
                          " (expert GEMM1+SwiGLU and GEMM2, one launch each per step; times "
                          "from the timed steps)",
                          "traffic": gemm_traffic(w),
                          "traffic_unit": "DRAM bytes per step (both GEMM launches), one ncu "
                                          "capture"}, **roof),
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * sx,
                "d2h_bytes_per_step": w.T * w.d * sx,
                "pipeline": "pinned host x -> device, layer, device y -> pinned host every "
                            "step; step i+1's upload and step i-1's download overlap step "
                            "i's layer (3 streams)"},
        "gpu_launches": len(r["stages"]) * args.steps,
        "launch": "programmatic dependent launch; events only around the expert GEMMs",
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
        "stats": {"kept_pairs": float(st[0]), "max_over_mean": float(st[4]),
                  "drop_fraction": float(st[5]), "balance": float(st[6]),
                  "balance_times_N": float(st[7])},
    }
    if w.mode == W.EXPERT_CHOICE:
        line["coverage"] = coverage_summary(r["coverage"])
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)


def run_stage(args):
    """--kernel STAGE: loop one stage of the layer on the workload (T
    overridable with --T) and print its device time and algorithmic GB/s.
    Holds only the routing-side tensors on the device (plus the routed
    experts for --kernel ffn, the expert FFN of the routed rows: both grouped
    GEMMs), so a single kernel can be profiled with ncu on inputs larger than
    L2."""
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = W.ALL[args.workload]
    if args.T:
        w = w.replace(T=args.T)
    inp = W.make_inputs(w, with_experts=args.kernel == "ffn")
    if w.weights == "e4m3":
        inp = {k: v for k, v in inp.items() if k not in ("W1", "W3", "W2")}
    d = {k: (v.to(dev) if v is not None and k not in ("Ws1", "Ws3", "Ws2") else None)
         for k, v in inp.items()}
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
    if args.kernel == "ffn":
        fsz = M.ffn_workspace_size_e4m3(R, w.d, w.f) if w.weights == "e4m3" else \
            M.ffn_workspace_size(R, w.f, w.dtype)
        fws = torch.zeros(fsz, dtype=torch.uint8, device=dev)
        if w.weights == "e4m3":
            ex = M.e4m3_experts(d["W1q"], d["W3q"], d["W2q"], d["W1s"], d["W3s"], d["W2s"])
            fns["ffn"] = lambda: M.moe_expert_ffn_e4m3(cfg, xp, offs, w.N, R, w.f, ex, op, fws)
        elif args.gather == "fused":
            fns["ffn"] = lambda: M.moe_expert_ffn_gather(cfg, d["x"], row_token, offs, w.N, R, w.f,
                                                         d["W1"], d["W3"], d["W2"], op, fws)
        else:
            fns["ffn"] = lambda: M.moe_expert_ffn(cfg, xp, offs, w.N, R, w.f, d["W1"], d["W3"],
                                                  d["W2"], op, fws)
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
    if args.kernel == "ffn":  # weights of the experts hit, rows in and out of both GEMMs
        nbytes = routed_weight_bytes(w, kept.cpu().numpy()) + \
            2 * P * (w.d + w.f) * (2 if w.dtype == "bf16" else 4)
    peaks, src = load_peaks()
    out = {"kernel": args.kernel, "workload": w.describe(), "kept_pairs": P, "ms": ms}
    if nbytes:
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.update({"bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / float(peaks["hbm_gbs"]),
                    "peak_source": src})
    print(json.dumps(out), flush=True)


# (segments, rows per segment, K, n_out): the Mixtral-shaped expert GEMMs at
# 1024 rows per expert (GEMM1 as one plain GEMM of width 2f, then GEMM2), and
# GEMM1's width on 614-row segments, whose last tiles are ragged
VS_CUBLAS_SHAPES = [(8, 1024, 4096, 28672), (8, 1024, 14336, 4096), (8, 614, 4096, 28672)]


def run_vs_cublas(args):
    """--vs-cublas: the plain grouped GEMM (moe_grouped_gemm, bf16) against
    cuBLAS's batched GEMM (torch.bmm) on the same equal-sized segments, the
    L2 flushed before every launch; prints both rates and the largest
    difference between the two outputs. A library yardstick for the expert
    GEMMs, not part of the layer."""
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    gen = torch.Generator(device=dev).manual_seed(7)

    def timed(fn):
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    rows_out = []
    for S, n, K, n_out in VS_CUBLAS_SHAPES:
        R = S * n
        A = (torch.randn((R, K), device=dev, generator=gen) * 0.05).to(torch.bfloat16)
        B = (torch.randn((S, K, n_out), device=dev, generator=gen) * 0.05).to(torch.bfloat16)
        out = torch.empty((R, n_out), dtype=torch.bfloat16, device=dev)
        ref = torch.empty_like(out)
        offs = torch.arange(0, R + 1, n, dtype=torch.int32, device=dev)
        ws = torch.zeros(M.ffn_workspace_size(0, 0, "bf16"), dtype=torch.uint8, device=dev)
        ms_ours = timed(lambda: M.moe_grouped_gemm("bf16", A, offs, S, R, K, n_out, B, out, ws))
        ms_lib = timed(lambda: torch.bmm(A.view(S, n, K), B, out=ref.view(S, n, n_out)))
        flops = 2.0 * R * K * n_out
        rows_out.append({"segments": S, "rows_per_segment": n, "K": K, "n_out": n_out,
                         "ours_ms": ms_ours, "ours_tflops": flops / (ms_ours * 1e-3) / 1e12,
                         "cublas_ms": ms_lib, "cublas_tflops": flops / (ms_lib * 1e-3) / 1e12,
                         "ours_over_cublas": ms_lib / ms_ours,
                         "max_abs_diff": (out.float() - ref.float()).abs().max().item()})
        del A, B, out, ref
    print(json.dumps({"metric": "grouped GEMM against cuBLAS batched GEMM", "unit": "TFLOP/s",
                      "steps": args.steps, "warmup": args.warmup,
                      "l2": "flushed before every launch", "rows": rows_out}), flush=True)


def run_ep_sim(args):
    """--ep-sim: expert parallelism simulated on one GPU ("Capacity-Aware
    Inference", section 1: under expert parallelism the layer waits for the
    most loaded device). The experts are split into `devices` groups of
    consecutive experts; after one routed layer step, each group's expert FFN
    runs alone on sm_count // devices SMs (moe_expert_ffn_on_sms) and is timed
    with CUDA events. The straggler time is the maximum over groups. The
    all-to-all exchange and the shared expert (the same on every device) are
    not part of the timing, and each group runs alone, so it does not share
    HBM with the others as it would inside one GPU."""
    import routing_capacity_drop_router_b300 as M
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    devices = args.ep_devices
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    per = sms // devices
    inf = math.inf
    cases = [(W.MIXTRAL_BF16, dict(mode=W.CAPACITY_DROP, gamma=g)) for g in (inf, 2.0, 1.5, 1.0)]
    fine = W.FINE_BF16
    cases += [(fine, dict(mode=W.CAPACITY_DROP, gamma=g)) for g in (inf, 1.5, 1.25, 1.0)]
    cases += [(fine, dict(mode=W.CAPACITY_DROP, gamma=1.25, m=4, group_size=fine.N // devices)),
              (fine, dict(mode=W.CAPACITY_DROP_DEVICE, gamma=1.25, group_size=fine.N // devices))]
    rows, inputs = [], {}
    for base, kw in cases:
        w = base.replace(name=base.name + "_epsim", **kw)
        if base.name not in inputs:
            inputs.clear()
            inp = W.make_inputs(base)
            inputs[base.name] = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
        d = inputs[base.name]
        cfg = M.config_from_workload(w)
        sz = M.sizes(cfg)
        ws = torch.zeros(sz.workspace, dtype=torch.uint8, device=dev)
        y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=dev)
        M.moe_layer_forward(cfg, d["x"], d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"],
                            d.get("Ws1"), d.get("Ws3"), d.get("Ws2"), y, ws)
        torch.cuda.synchronize()
        v = M.moe_workspace_views(cfg, ws)
        k0 = v.kept - ws.data_ptr()  # the per-expert kept counts live in the workspace
        kept_h = ws[k0:k0 + 4 * w.N].view(torch.int32).cpu().numpy()
        gs = w.N // devices
        fws = torch.zeros(M.ffn_workspace_size(sz.rows_max, w.f, w.dtype), dtype=torch.uint8,
                          device=dev)
        times = []
        for g in range(devices):
            lo = g * gs
            call = lambda: M.moe_expert_ffn_on_sms(
                cfg, v.xp, v.expert_offsets + 4 * lo, gs, sz.rows_max, w.f,
                d["W1"][lo].data_ptr(), d["W3"][lo].data_ptr(), d["W2"][lo].data_ptr(), v.op,
                per, fws)
            for _ in range(2):
                call()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.ep_reps)]
            for a, b in evs:
                a.record()
                call()
                b.record()
            torch.cuda.synchronize()
            times.append(statistics.median(a.elapsed_time(b) for a, b in evs))
        if M.moe_get_device_status(fws) != M.MOE_OK:
            raise RuntimeError("device status error in the expert-parallel simulation")
        loads = [int(kept_h[g * gs:(g + 1) * gs].sum()) for g in range(devices)]
        rows.append({"workload": base.name, "mode": w.mode,
                     "gamma": None if math.isinf(w.gamma) else w.gamma, "m": w.m,
                     "device_loads": loads,
                     "max_over_mean_load": max(loads) / (sum(loads) / devices),
                     "straggler_ms": max(times), "mean_device_ms": sum(times) / devices,
                     "device_ms": [round(t, 4) for t in times]})
        del ws, fws
    for r in rows:  # speed-up of the straggler against the same layer without a capacity
        ref = next(q for q in rows if q["workload"] == r["workload"] and q["gamma"] is None)
        r["straggler_speedup_vs_no_capacity"] = ref["straggler_ms"] / r["straggler_ms"]
    print(json.dumps({"metric": "simulated expert-parallel straggler time of the routed experts",
                      "unit": "ms", "higher_is_better": False, "devices": devices,
                      "sms_per_device": per, "reps": args.ep_reps, "rows": rows}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.ALL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline workload only (skip the line's \"configs\" object)")
    ap.add_argument("--cpu-sample-s", type=float, default=15.0,
                    help="seconds of oracle work in the cpu_baseline sample")
    ap.add_argument("--reference-budget-s", type=float, default=150.0,
                    help="--impl reference: seconds for warm-up + timed samples together")
    ap.add_argument("--distinct-batches", action="store_true",
                    help="each rank draws its own x (seed + rank)")
    ap.add_argument("--kernel", choices=["route", "select", "dispatch", "combine", "ffn"],
                    help="time one stage alone instead of the layer")
    ap.add_argument("--T", type=int, default=0, help="token count override for --kernel")
    ap.add_argument("--gather", choices=["copy", "fused"], default="copy",
                    help="bf16 experts: dispatch copies the token rows (copy) or expert GEMM1 "
                         "gathers them itself (fused, MOE_FUSE_GATHER)")
    ap.add_argument("--ep-sim", action="store_true",
                    help="simulate expert parallelism: time each device group's experts on "
                         "its share of the SMs and report the straggler")
    ap.add_argument("--vs-cublas", action="store_true",
                    help="time the plain grouped GEMM beside cuBLAS's batched GEMM on the "
                         "same segments")
    ap.add_argument("--ep-devices", type=int, default=8)
    ap.add_argument("--ep-reps", type=int, default=10)
    args = ap.parse_args()
    if args.kernel:
        run_stage(args)
        return
    if args.ep_sim:
        run_ep_sim(args)
        return
    if args.vs_cublas:
        run_vs_cublas(args)
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
