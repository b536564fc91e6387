"""Whole-layer GPU parity (moe_layer_forward) against the oracle.

Small shapes run every token through the oracle; they span several 128-row
tiles with ragged tails. The benchmark workloads run at full size with the
oracle computing a sample of tokens (a token's output depends only on its own
routing, which the oracle computes for the whole batch), in the launch
configuration the benchmark times."""
import math

import numpy as np
import pytest
import torch

import moe_workloads as W
import oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SMALL = [
    W.Workload("small_tc", T=600, d=256, N=8, f=384, k=2),
    W.Workload("small_drop_renorm", T=600, d=256, N=8, f=384, k=2, mode=W.CAPACITY_DROP,
               gamma=1.0, renorm=True, zipf_s=1.2),
    W.Workload("small_ec", T=640, d=192, N=8, f=256, k=2, mode=W.EXPERT_CHOICE),
    W.Workload("small_expanded_shared", T=500, d=128, N=16, f=128, k=3, mode=W.CAPACITY_DROP,
               gamma=1.25, m=2, group_size=4, f_shared=192, zipf_s=1.0),
    W.Workload("small_f32", T=300, d=64, N=4, f=96, k=2, dtype="f32", mode=W.CAPACITY_DROP,
               gamma=1.0),
    W.Workload("small_device_shared", T=500, d=128, N=16, f=128, k=3,
               mode=W.CAPACITY_DROP_DEVICE, gamma=1.0, group_size=4, f_shared=192, zipf_s=1.0),
    W.Workload("small_drop_e4m3_shared", T=600, d=256, N=8, f=384, k=2, mode=W.CAPACITY_DROP,
               gamma=1.0, renorm=True, zipf_s=1.2, f_shared=128, weights="e4m3"),
]


def _check_layer(w, inp, tokens=None):
    # 1) both sides given the oracle's fp32 logits: routing identical, y within tolerance
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    ref = G.oracle_layer(w, inp, logits=L, tokens=tokens)
    got = G.layer_gpu(w, inp, logits=L, want_views=True)
    assert np.array_equal(got["kept"], ref["kept"])
    assert np.array_equal(got["keep"].astype(bool), ref["keep"])
    assert np.array_equal(got["coverage"], ref["coverage"])
    rows = ref["tokens"]
    G.assert_output_close(got["y"][rows], ref["y"], w.dtype)
    s = O.load_stats(ref["demand"], ref["kept"], ref["p"])
    want = [s["P"], s["demand_total"], s["max_kept"], s["mean_kept"], s["max_over_mean"],
            s["drop_fraction"], s["balance"], s["balance_times_N"]]
    assert np.allclose(got["stats"], want, rtol=1e-5, atol=1e-9)
    return L, ref, got


def _check_own_logits(w, inp, L, ref, tokens=None):
    # 2) the GPU computes its own logits: within the fp32 bound of the oracle's;
    # tokens whose routing is unchanged match the oracle's output
    got = G.layer_gpu(w, inp, want_views=True)
    bound = G.logit_bound(G.np32(inp["x"]), G.np32(inp["W_r"]), L)
    assert np.all(np.abs(got["logits"].astype(np.float64) - L) <= bound)
    rows = ref["tokens"]
    same = np.all(got["keep"].astype(bool)[rows] == ref["keep"][rows], axis=1)
    if w.mode != W.EXPERT_CHOICE:
        same &= np.all(got["cand_idx"][rows] == ref["idx"][rows], axis=1)
    assert same.mean() >= 0.99, f"{(~same).sum()} of {len(rows)} tokens routed differently"
    G.assert_output_close(got["y"][rows][same], ref["y"][same], w.dtype)


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_layer_parity(w):
    inp = W.make_inputs(w)
    L, ref, _ = _check_layer(w, inp)
    _check_own_logits(w, inp, L, ref)


def test_tiny_fp32_workload_full():
    w = W.TINY_F32
    inp = W.make_inputs(w)
    L, ref, _ = _check_layer(w, inp)
    _check_own_logits(w, inp, L, ref)


FUSABLE = [w for w in SMALL if w.dtype == "bf16" and w.weights == "same"]


@pytest.mark.parametrize("w", FUSABLE, ids=[w.name for w in FUSABLE])
def test_small_layer_fused_gather(w):
    """MOE_FUSE_GATHER: GEMM1 reads the token rows through row_token; the
    layer output is the same bits as with the dispatched copy, and within
    tolerance of the oracle."""
    inp = W.make_inputs(w)
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    ref = G.oracle_layer(w, inp, logits=L)
    copy = G.layer_gpu(w, inp, logits=L)
    fused = G.layer_gpu(w, inp, logits=L, fuse_gather=True, want_views=True)
    assert np.array_equal(fused["y"], copy["y"])
    assert np.array_equal(fused["kept"], ref["kept"])
    G.assert_output_close(fused["y"][ref["tokens"]], ref["y"], w.dtype)


@pytest.mark.parametrize("name", ["mixtral_bf16_gamma1", "expert_choice_bf16",
                                  "finegrained_bf16_expanded"])
def test_fused_gather_full_size(name):
    """The benchmark workloads at full size with MOE_FUSE_GATHER: the same
    output bits as the copy path, and a token sample within tolerance of the
    oracle."""
    w = W.ALL[name]
    inp = W.make_inputs(w)
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    copy = G.layer_gpu(w, inp, logits=L)
    fused = G.layer_gpu(w, inp, logits=L, fuse_gather=True)
    assert np.array_equal(fused["y"], copy["y"])
    tokens = np.union1d(np.random.default_rng(1).choice(w.T, size=16, replace=False),
                        G.tile_edge_tokens(w, L))
    ref = G.oracle_layer(w, inp, logits=L, tokens=tokens)
    G.assert_output_close(fused["y"][ref["tokens"]], ref["y"], w.dtype)


DEGENERATE = [
    W.Workload("one_token_top1", T=1, d=128, N=8, f=128, k=1),
    W.Workload("one_token_no_room", T=1, d=128, N=8, f=128, k=2, mode=W.CAPACITY_DROP,
               gamma=1.0),  # C = floor(1.0 * 2 * 1 / 8) = 0: the token is dropped everywhere
    W.Workload("every_expert", T=300, d=128, N=8, f=128, k=8, renorm=True),  # dense mixture
    W.Workload("every_expert_choice", T=64, d=128, N=8, f=128, k=8,
               mode=W.EXPERT_CHOICE),  # c = T: each expert takes every token
    # the limits: 256 experts (one GEMM segment each), 32 candidate slots per token
    W.Workload("max_experts", T=300, d=64, N=256, f=64, k=8, mode=W.CAPACITY_DROP, gamma=1.0),
    W.Workload("max_slots", T=200, d=64, N=64, f=64, k=24, m=8, group_size=16,
               mode=W.CAPACITY_DROP, gamma=1.25),
    # the fp32 path (FMA GEMMs; the fused-gather flag does not apply to it)
    W.Workload("one_token_f32", T=1, d=64, N=8, f=96, k=2, dtype="f32"),
    W.Workload("max_experts_f32", T=300, d=64, N=256, f=64, k=8, mode=W.CAPACITY_DROP,
               gamma=1.0, dtype="f32"),
]


@pytest.mark.parametrize("fuse", [False, True], ids=["copy", "fused_gather"])
@pytest.mark.parametrize("w", DEGENERATE, ids=[w.name for w in DEGENERATE])
def test_degenerate_layers(w, fuse):
    """The method's degenerate cases through the whole layer (one token, no
    room at all, every expert per token under token and expert choice) and
    its limits (256 experts, 32 candidate slots)."""
    inp = W.make_inputs(w)
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    ref = G.oracle_layer(w, inp, logits=L)
    got = G.layer_gpu(w, inp, logits=L, want_views=True, fuse_gather=fuse)
    assert np.array_equal(got["kept"], ref["kept"])
    G.assert_output_close(got["y"], ref["y"], w.dtype)


@pytest.mark.parametrize("w", [
    W.Workload("repeat_drop_expanded_shared", T=3000, d=256, N=64, f=128, k=6, m=2,
               group_size=8, mode=W.CAPACITY_DROP, gamma=1.25, f_shared=128, zipf_s=1.0),
    W.Workload("repeat_device", T=3000, d=256, N=64, f=128, k=6, group_size=8,
               mode=W.CAPACITY_DROP_DEVICE, gamma=1.0, zipf_s=1.0),
    W.Workload("repeat_ec", T=2048, d=256, N=16, f=128, k=2, mode=W.EXPERT_CHOICE),
], ids=lambda w: w.name)
def test_repeated_calls_on_one_workspace_are_bitwise_identical(w):
    """Five back-to-back layer calls (own router logits) on one workspace that
    is never re-zeroed: every call leaves the control block as it found it and
    nothing depends on the order of atomics, so logits, y and the statistics
    repeat bit for bit."""
    inp = W.make_inputs(w)
    cfg = G.M.config_from_workload(w)
    dev = torch.device("cuda")
    ws = torch.zeros(G.M.workspace_size(cfg), dtype=torch.uint8, device=dev)
    d = {k: G.cuda(inp.get(k)) for k in ("x", "W_r", "bias", "W1", "W3", "W2", "Ws1", "Ws3", "Ws2")}
    outs = []
    for _ in range(5):
        y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=dev)
        L = torch.empty((w.T, w.N), dtype=torch.float32, device=dev)
        st = torch.zeros(G.M.MOE_STATS_LEN, dtype=torch.float64, device=dev)
        G.M.moe_layer_forward(cfg, d["x"], d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"],
                              d["Ws1"], d["Ws3"], d["Ws2"], y, ws, logits=L, stats=st)
        outs.append((y, L, st))
    torch.cuda.synchronize()
    assert G.M.moe_get_device_status(ws) == G.M.MOE_OK
    y0, L0, s0 = outs[0]
    for y, L, st in outs[1:]:
        assert torch.equal(L, L0) and torch.equal(y, y0) and torch.equal(st, s0)
    assert s0[0].item() > 0


def test_empty_layer():
    """T = 0 through the whole layer: nothing routed, nothing written, no error."""
    w = W.Workload("empty_layer", T=0, d=128, N=8, f=128, k=2, mode=W.CAPACITY_DROP, gamma=1.0)
    inp = W.make_inputs(w)
    got = G.layer_gpu(w, inp, want_views=True)
    assert got["y"].shape == (0, w.d)
    assert (got["kept"] == 0).all()
    assert got["stats"][0] == 0


def test_capacity_zero_outputs_zero():
    w = W.Workload("zero_cap", T=200, d=128, N=8, f=128, k=2, mode=W.CAPACITY_DROP, gamma=0.0)
    inp = W.make_inputs(w)
    got = G.layer_gpu(w, inp)
    assert np.all(got["y"] == 0)
    assert got["stats"][0] == 0 and got["stats"][5] == 1.0


def test_gamma_inf_equals_token_choice_bitwise():
    w_tc = W.Workload("tc", T=400, d=128, N=8, f=128, k=2, renorm=True)
    w_drop = w_tc.replace(name="drop_inf", mode=W.CAPACITY_DROP, gamma=math.inf)
    inp = W.make_inputs(w_tc)
    a = G.layer_gpu(w_tc, inp)
    b = G.layer_gpu(w_drop, inp)
    assert np.array_equal(a["y"], b["y"])


@pytest.mark.slow
@pytest.mark.parametrize("name,sample", [
    ("expert_choice_bf16", None),
    ("decode_bf16", None),
    ("mixtral_bf16_gamma1", 48),
    ("mixtral_bf16", 32),
    ("finegrained_bf16", 64),
    ("finegrained_bf16_expanded", 64),
    ("finegrained_bf16_device", 64),
    ("decode_e4m3", None),
])
def test_benchmark_workloads_full_size(name, sample):
    """Full size. Sampled workloads check a random token sample plus every
    token at the first or last row of a 128-row tile of an expert segment, so
    that every tile of both GEMMs is checked at the full d and f depth."""
    w = W.ALL[name]
    inp = W.make_inputs(w)
    tokens = None
    if sample is not None:
        rng = np.random.default_rng(0)
        L0 = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
        tokens = np.union1d(rng.choice(w.T, size=sample, replace=False),
                            G.tile_edge_tokens(w, L0))
    L, ref, _ = _check_layer(w, inp, tokens=tokens)
    _check_own_logits(w, inp, L, ref, tokens=tokens)


def test_trace_events_time_every_stage():
    """moe_set_trace_events: one event before the first kernel and one after
    each stage, in launch order, on the call's stream."""
    w = SMALL[3]  # expanded drop + shared expert: the longest stage list
    inp = W.make_inputs(w)
    cfg = G.M.config_from_workload(w)
    names = G.M.moe_layer_stages(cfg)
    d = {k: G.cuda(v) for k, v in inp.items()}
    ws = torch.zeros(G.M.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    stats = torch.zeros(G.M.MOE_STATS_LEN, dtype=torch.float64, device="cuda")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    G.M.moe_set_trace_events(evs)
    try:
        G.M.moe_layer_forward(cfg, d["x"], d["W_r"], d["bias"], d["W1"], d["W3"], d["W2"],
                              d["Ws1"], d["Ws3"], d["Ws2"], y, ws, stats=stats)
    finally:
        G.M.moe_set_trace_events(None)
    torch.cuda.synchronize()
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(names))]
    assert all(m >= 0 for m in ms)
    assert evs[0].elapsed_time(evs[-1]) > 0
    assert G.M.moe_get_device_status(ws) == G.M.MOE_OK
