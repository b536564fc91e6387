"""The layer through its split C-ABI calls, in the order a caller would chain
them: moe_route (given logits) -> moe_capacity_drop -> moe_dispatch ->
moe_expert_ffn (routed experts, then the shared expert on the token rows) ->
moe_combine, plus moe_load_stats. The same kernels run as in
moe_layer_forward, so y must equal the fused call's bit for bit, and the
statistics must equal the fused call's; y is also checked against the
oracle."""
import numpy as np
import pytest
import torch

import moe_workloads as W
import oracle as O
from tests import gpu_util as G

M = G.M
pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("split_expanded_shared", T=500, d=128, N=16, f=128, k=3, mode=W.CAPACITY_DROP,
               gamma=1.25, m=2, group_size=4, f_shared=192, zipf_s=1.0),
    W.Workload("split_ec", T=640, d=192, N=8, f=256, k=2, mode=W.EXPERT_CHOICE),
    W.Workload("split_f32_drop", T=300, d=64, N=4, f=96, k=2, dtype="f32", mode=W.CAPACITY_DROP,
               gamma=1.0),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_split_calls_equal_the_fused_layer(w):
    inp = W.make_inputs(w)
    L = O.router_logits(G.np32(inp["x"]), G.np32(inp["W_r"]), G.np32(inp["bias"]))
    cfg = M.config_from_workload(w, logits_given=True)
    sz = M.sizes(cfg)
    T, N, kc, R = w.T, w.N, sz.kc, int(sz.rows_max)
    dev = torch.device("cuda")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    f32, i32 = torch.float32, torch.int32
    d = {k: G.cuda(v) for k, v in inp.items()}
    Ld = torch.from_numpy(np.ascontiguousarray(L)).to(dev)
    ec = w.mode == W.EXPERT_CHOICE

    scores = torch.empty((T, N), dtype=f32, device=dev)
    cand_idx = torch.empty((T, kc), dtype=i32, device=dev)
    cand_gate = torch.empty((T, kc), dtype=f32, device=dev)
    rws = torch.zeros(M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    M.moe_route(cfg, None, None, None, Ld, scores, None if ec else cand_idx, cand_gate, rws)
    slot = torch.empty((T, kc), dtype=i32, device=dev)
    keep = torch.empty((T, kc), dtype=torch.uint8, device=dev)
    demand = torch.empty((N,), dtype=i32, device=dev)
    kept = torch.empty((N,), dtype=i32, device=dev)
    M.moe_capacity_drop(cfg, None if ec else cand_idx, cand_gate, slot, keep, demand, kept)
    offs = torch.empty((N + 1,), dtype=i32, device=dev)
    row_token = torch.empty((R,), dtype=i32, device=dev)
    row_gate = torch.empty((R,), dtype=f32, device=dev)
    tok_rows = torch.empty((T, kc), dtype=i32, device=dev)
    coverage = torch.empty((T,), dtype=i32, device=dev)
    xp = torch.zeros((R, w.d), dtype=dt, device=dev)
    M.moe_dispatch(cfg, d["x"], None if ec else cand_idx, cand_gate, slot, kept, offs, row_token,
                   row_gate, tok_rows, xp, coverage=coverage)
    op = torch.zeros((R, w.d), dtype=dt, device=dev)
    fws = torch.zeros(M.ffn_workspace_size(R, w.f, w.dtype), dtype=torch.uint8, device=dev)
    M.moe_expert_ffn(cfg, xp, offs, N, R, w.f, d["W1"], d["W3"], d["W2"], op, fws)
    ys = None
    if w.f_shared:  # the shared expert: one segment of all T token rows
        soff = torch.tensor([0, T], dtype=i32, device=dev)
        ys = torch.empty((T, w.d), dtype=dt, device=dev)
        sws = torch.zeros(M.ffn_workspace_size(T, w.f_shared, w.dtype), dtype=torch.uint8,
                          device=dev)
        M.moe_expert_ffn(cfg, d["x"], soff, 1, T, w.f_shared, d["Ws1"], d["Ws3"], d["Ws2"], ys,
                         sws)
    y = torch.empty((T, w.d), dtype=dt, device=dev)
    M.moe_combine(cfg, op, row_gate, tok_rows, ys, y)
    stats = torch.zeros(M.MOE_STATS_LEN, dtype=torch.float64, device=dev)
    stws = torch.zeros(8 * N * -(-T // 32), dtype=torch.uint8, device=dev)  # column sums
    M.moe_load_stats(cfg, demand, kept, scores, stats, stws)
    torch.cuda.synchronize()
    for ws in (rws, fws):
        assert M.moe_get_device_status(ws) == M.MOE_OK

    fused = G.layer_gpu(w, inp, logits=L, want_views=True)
    assert np.array_equal(G.np32(y), fused["y"]), "split calls and the fused layer differ"
    assert np.array_equal(coverage.cpu().numpy(), fused["coverage"])
    assert np.array_equal(stats.cpu().numpy(), fused["stats"])
    ref = G.oracle_layer(w, inp, logits=L)
    G.assert_output_close(G.np32(y), ref["y"], w.dtype)
