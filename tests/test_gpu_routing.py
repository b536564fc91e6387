"""GPU routing parity: scores, top-k / expanded candidates, gates, per-expert
selection (capacity drop, expert choice), offsets, row maps and token rows
must equal the oracle's bit for bit when both get the same fp32 logits; the
GPU's own router logits must sit within the fp32 accumulation bound."""
import math

import numpy as np
import pytest
import torch

import moe_workloads as W
import oracle as O
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _logits_of(w):
    inp = W.make_inputs(w, with_experts=False)
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    return inp, L


@pytest.mark.parametrize("name", list(W.ALL))
def test_routing_bit_exact_on_every_workload(name):
    w = W.ALL[name]
    inp, L = _logits_of(w)
    g = G.gpu_routing(w, torch.from_numpy(L), x=inp["x"])
    G.compare_routing(w, g, L)
    # the gather: every used row of xp is its token's row of x, bitwise
    P = int(g["expert_offsets"][-1])
    xp = g["xp"][:P]
    assert torch.equal(xp, inp["x"][torch.from_numpy(g["row_token"][:P]).long()])


SMALL = [
    W.Workload("tc_ties", T=1000, d=64, N=16, f=64, k=4),
    W.Workload("drop_ties", T=1000, d=64, N=16, f=64, k=4, mode=W.CAPACITY_DROP, gamma=1.0),
    W.Workload("drop_renorm_ties", T=777, d=64, N=8, f=64, k=2, mode=W.CAPACITY_DROP,
               gamma=0.75, renorm=True),
    W.Workload("ec_ties", T=999, d=64, N=16, f=64, k=3, mode=W.EXPERT_CHOICE),
    W.Workload("expanded_ties", T=1001, d=64, N=32, f=64, k=3, mode=W.CAPACITY_DROP, gamma=1.0,
               m=3, group_size=4),
    W.Workload("drop_zero_capacity", T=100, d=64, N=8, f=64, k=2, mode=W.CAPACITY_DROP, gamma=0.0),
    W.Workload("ec_c_equals_T", T=64, d=64, N=4, f=64, k=4, mode=W.EXPERT_CHOICE),
    W.Workload("one_expert", T=300, d=64, N=1, f=64, k=1),
    W.Workload("many_experts", T=513, d=64, N=256, f=64, k=8, mode=W.CAPACITY_DROP, gamma=1.0),
    W.Workload("ec_many_experts", T=300, d=64, N=64, f=64, k=2, mode=W.EXPERT_CHOICE),
    # device-level capacity ("Capacity-Aware Inference", section 2 (3))
    W.Workload("device_ties", T=1000, d=64, N=16, f=64, k=4, mode=W.CAPACITY_DROP_DEVICE,
               gamma=1.0, group_size=4),
    W.Workload("device_expanded_renorm", T=1001, d=64, N=32, f=64, k=3,
               mode=W.CAPACITY_DROP_DEVICE, gamma=0.8, m=3, group_size=8, renorm=True),
    W.Workload("device_one_expert_each", T=777, d=64, N=8, f=64, k=2,
               mode=W.CAPACITY_DROP_DEVICE, gamma=0.75, group_size=1),
    W.Workload("device_single_group", T=513, d=64, N=16, f=64, k=4, mode=W.CAPACITY_DROP_DEVICE,
               gamma=0.5, group_size=16),
    W.Workload("device_zero_capacity", T=100, d=64, N=8, f=64, k=2, mode=W.CAPACITY_DROP_DEVICE,
               gamma=0.0, group_size=4),
    W.Workload("device_max_tokens", T=24576, d=64, N=64, f=64, k=8, mode=W.CAPACITY_DROP_DEVICE,
               gamma=1.0, group_size=8),
    W.Workload("device_group_of_32", T=3000, d=64, N=64, f=64, k=4, mode=W.CAPACITY_DROP_DEVICE,
               gamma=0.8, group_size=32),  # larger than a cluster: table passes
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
@pytest.mark.parametrize("quantum", [None, 0.25])
def test_routing_bit_exact_with_ties_and_ragged_sizes(w, quantum):
    L = W.random_logits(w.T, w.N, seed=3, scale=2.0, quantum=quantum)
    g = G.gpu_routing(w, L)
    G.compare_routing(w, g, L.numpy())


def test_all_equal_logits_and_signed_zeros():
    w = W.Workload("flat", T=257, d=64, N=8, f=64, k=3, mode=W.CAPACITY_DROP, gamma=1.0)
    L = torch.zeros((w.T, w.N))
    L[::2, ::3] = -0.0
    g = G.gpu_routing(w, L)
    G.compare_routing(w, g, L.numpy())
    assert (g["cand_idx"] == np.array([0, 1, 2])).all()


@pytest.mark.parametrize("gs", [4, 16])
def test_device_drop_with_every_gate_equal(gs):
    """All logits equal: every token's candidates are the lowest experts with
    equal gates, so one device holds thousands of ties (more than a CTA's tie
    list) and the kept set is decided by (token, slot) order alone."""
    w = W.Workload("device_flat", T=12000, d=64, N=16, f=64, k=2, mode=W.CAPACITY_DROP_DEVICE,
                   gamma=0.5, group_size=gs)
    L = torch.zeros((w.T, w.N))
    g = G.gpu_routing(w, L)
    G.compare_routing(w, g, L.numpy())
    assert 0 < g["keep"].sum() < w.T * 2


def test_given_home_groups():
    w = W.Workload("home", T=300, d=64, N=16, f=64, k=2, mode=W.CAPACITY_DROP, gamma=1.0, m=2,
                   group_size=4)
    L = W.random_logits(w.T, w.N, seed=5)
    hg = torch.from_numpy(np.random.default_rng(5).integers(0, 4, size=w.T).astype(np.int32))
    g = G.gpu_routing(w, L, home_group=hg)
    G.compare_routing(w, g, L.numpy(), home_group=hg.numpy())


def test_empty_batch():
    w = W.Workload("empty", T=0, d=64, N=8, f=64, k=2, mode=W.CAPACITY_DROP, gamma=1.0)
    g = G.gpu_routing(w, torch.zeros((0, 8)))
    assert (g["demand"] == 0).all() and (g["kept"] == 0).all()
    assert (g["expert_offsets"] == 0).all()


@pytest.mark.parametrize("name", ["tiny_fp32", "expert_choice_bf16", "mixtral_bf16",
                                  "finegrained_bf16", "decode_bf16"])
def test_router_logits_within_fp32_bound(name):
    w = W.ALL[name]
    inp, L = _logits_of(w)
    cfg = G.M.config_from_workload(w)
    sz = G.M.sizes(cfg)
    dev = torch.device("cuda")
    Lg = torch.empty((w.T, w.N), dtype=torch.float32, device=dev)
    idx = torch.empty((w.T, sz.kc), dtype=torch.int32, device=dev)
    gate = torch.empty((w.T, sz.kc), dtype=torch.float32, device=dev)
    rws = torch.zeros(G.M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    G.M.moe_route(cfg, G.cuda(inp["x"]), G.cuda(inp["W_r"]), G.cuda(inp["bias"]), Lg, None,
                  None if w.mode == W.EXPERT_CHOICE else idx, gate, rws)
    torch.cuda.synchronize()
    diff = np.abs(Lg.cpu().numpy().astype(np.float64) - L.astype(np.float64))
    bound = G.logit_bound(G.np32(inp["x"]), G.np32(inp["W_r"]), L)
    assert np.all(diff <= bound), float((diff / bound).max())


def _route_own_logits(w, inp, rws=None):
    """moe_route with the router computing its own logits (on bf16 layers the
    tensor-core router, which routes each tile in its last CTA)."""
    cfg = G.M.config_from_workload(w)
    sz = G.M.sizes(cfg)
    dev = torch.device("cuda")
    Lg = torch.empty((w.T, w.N), dtype=torch.float32, device=dev)
    scores = torch.empty((w.T, w.N), dtype=torch.float32, device=dev)
    idx = torch.full((w.T, sz.kc), -7, dtype=torch.int32, device=dev)
    gate = torch.full((w.T, sz.kc), -7.0, dtype=torch.float32, device=dev)
    if rws is None:
        rws = torch.zeros(G.M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    G.M.moe_route(cfg, G.cuda(inp["x"]), G.cuda(inp["W_r"]), G.cuda(inp["bias"]), Lg, scores,
                  None if w.mode == W.EXPERT_CHOICE else idx, gate, rws)
    torch.cuda.synchronize()
    return Lg.cpu().numpy(), scores.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy()


def _assert_routing_of(w, L, scores, idx, gate):
    rt = G.oracle_route(w, L)
    assert np.array_equal(scores.view(np.uint32), rt["p"].view(np.uint32)), "scores differ"
    if w.mode != W.EXPERT_CHOICE:
        assert np.array_equal(idx, rt["idx"]), "candidate experts differ"
    assert np.array_equal(gate.view(np.uint32), rt["gate"].view(np.uint32)), "gates differ"


@pytest.mark.parametrize("name", ["expert_choice_bf16", "mixtral_bf16_gamma1", "finegrained_bf16",
                                  "finegrained_bf16_expanded", "decode_bf16"])
def test_fused_router_routes_its_own_logits_bit_exactly(name):
    """The tensor-core router's in-kernel routing equals the oracle's routing
    of the logits that router produced."""
    w = W.ALL[name]
    inp = W.make_inputs(w, with_experts=False)
    _assert_routing_of(w, *_route_own_logits(w, inp))


def test_router_workspace_reused_across_shapes():
    """The router's per-tile arrival counters return to zero after every
    launch, so one workspace serves configs with different split counts."""
    big = W.Workload("reuse_big", T=1000, d=1024, N=16, f=64, k=2, zipf_s=1.0)
    small = W.Workload("reuse_small", T=300, d=256, N=8, f=64, k=2, mode=W.CAPACITY_DROP,
                       gamma=1.0)
    n = max(G.M.route_workspace_size(G.M.config_from_workload(v)) for v in (big, small))
    rws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for w in (big, small, big, small):
        inp = W.make_inputs(w, with_experts=False)
        _assert_routing_of(w, *_route_own_logits(w, inp, rws))
    ctrl = rws[:G.M.MOE_CTRL_BYTES].view(torch.int32).cpu().numpy()
    assert (ctrl == 0).all(), "control block not back at zero"


ROUTER_TAIL = [
    # one CTA per tile (3 k-blocks of 64 do not split in two): 128 tokens per
    # CTA, 256 experts, renormalised top-8
    W.Workload("tail_c1_n256", T=300, d=192, N=256, f=64, k=8, renorm=True, zipf_s=1.0),
    # 128 experts, expanded candidates from groups of 16, capacity drop
    W.Workload("tail_n128_expanded", T=1000, d=512, N=128, f=64, k=4, m=4, group_size=16,
               mode=W.CAPACITY_DROP, gamma=1.25),
    # N not a power of two, expert choice, ragged last tile
    W.Workload("tail_n24_ec", T=777, d=1024, N=24, f=64, k=3, mode=W.EXPERT_CHOICE),
]


@pytest.mark.parametrize("w", ROUTER_TAIL, ids=[w.name for w in ROUTER_TAIL])
def test_router_tail_shapes_bit_exact(w):
    """The router tail (partials summed in rank order, one thread per token)
    routes its own logits exactly as the oracle does, at the shapes where the
    tail's chunking and row rotation change: one CTA per tile, N = 256, N not
    a power of two, a ragged last tile."""
    inp = W.make_inputs(w, with_experts=False)
    L, scores, idx, gate = _route_own_logits(w, inp)
    bound = G.logit_bound(G.np32(inp["x"]), G.np32(inp["W_r"]),
                          O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]),
                                          G.np32(inp["bias"])))
    ref = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    assert np.all(np.abs(L.astype(np.float64) - ref) <= bound)
    _assert_routing_of(w, L, scores, idx, gate)


def test_router_tail_ties_bit_exact():
    """Integer-valued x and W_r make the logits exact and full of ties, so the
    tail's tie-breaks (lower expert first) decide most of the top-k."""
    w = W.Workload("tail_ties", T=513, d=256, N=64, f=64, k=6, renorm=True)
    g = torch.Generator().manual_seed(77)
    x = torch.randint(-1, 2, (w.T, w.d), generator=g).to(torch.bfloat16)
    W_r = (torch.randint(-1, 2, (w.d, w.N), generator=g).float() / 4).to(torch.bfloat16)
    inp = {"x": x, "W_r": W_r, "bias": None}
    L, scores, idx, gate = _route_own_logits(w, inp)
    ref = O.router_logits(G.np32(x), G.np32(W_r), None)
    assert np.array_equal(L, ref)  # exact: small integers times quarters
    assert (np.sort(L, axis=1)[:, 1:] == np.sort(L, axis=1)[:, :-1]).any(axis=1).mean() > 0.9
    _assert_routing_of(w, L, scores, idx, gate)
