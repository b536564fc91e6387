"""Helpers shared by the GPU parity tests: upload seeded inputs, run the
library's split entry points, and compare against the oracle."""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np
import torch

import moe_workloads as W
import oracle as O
import routing_capacity_drop_router_b300 as M

BF16_REL_FROB = 5e-3     # relative Frobenius error, bf16 in / fp32 accumulate
BF16_MAX_ABS = 1e-2      # max-abs error as a fraction of max |y_ref|
F32_REL_FROB = 1e-5      # fp32 layer: relative Frobenius error
F32_MAX_ABS = 1e-5       # fp32 layer: max-abs error as a fraction of max |y_ref|


def cuda(t: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    return None if t is None else t.contiguous().cuda()


def np32(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    return None if t is None else t.detach().float().cpu().numpy()


def rel_frob(y: np.ndarray, ref: np.ndarray) -> float:
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(y - ref) / den) if den > 0 else float(np.linalg.norm(y))


def assert_output_close(y: np.ndarray, ref: np.ndarray, dtype: str, what: str = "y") -> None:
    if dtype == "bf16":
        rf = rel_frob(y, ref)
        mx = float(np.max(np.abs(np.asarray(y, np.float64) - ref))) if ref.size else 0.0
        scale = float(np.max(np.abs(ref))) if ref.size else 0.0
        assert rf <= BF16_REL_FROB, f"{what}: relative Frobenius error {rf:.3e}"
        assert mx <= BF16_MAX_ABS * scale + 1e-30, f"{what}: max-abs error {mx:.3e} vs {scale:.3e}"
    else:
        # the 1e-5 relative bound, both as a norm and element by element
        rf = rel_frob(y, ref)
        mx = float(np.max(np.abs(np.asarray(y, np.float64) - ref))) if ref.size else 0.0
        scale = float(np.max(np.abs(ref))) if ref.size else 0.0
        assert rf <= F32_REL_FROB, f"{what}: relative Frobenius error {rf:.3e}"
        assert mx <= F32_MAX_ABS * scale + 1e-30, f"{what}: max-abs error {mx:.3e} vs {scale:.3e}"


def oracle_route(w: W.Workload, L: np.ndarray, home_group=None) -> Dict[str, np.ndarray]:
    return O.route(L, mode=w.mode, k=w.k, N=w.N, gamma=w.gamma, m=w.m,
                   group_size=w.group_size, renorm=w.renorm, home_group=home_group)


def gpu_routing(w: W.Workload, L: torch.Tensor, home_group: Optional[torch.Tensor] = None,
                x: Optional[torch.Tensor] = None) -> Dict[str, np.ndarray]:
    """Route -> select -> dispatch on the GPU from given fp32 logits; returns
    host copies of every output. With ``x`` also gathers xp."""
    cfg = M.config_from_workload(w, logits_given=True)
    sz = M.sizes(cfg)
    T, N, kc, R = w.T, w.N, sz.kc, max(int(sz.rows_max), 1)
    dev = torch.device("cuda")
    Ld = L.contiguous().to(dev)
    scores = torch.empty((T, N), dtype=torch.float32, device=dev)
    cand_idx = torch.full((T, kc), -7, dtype=torch.int32, device=dev)
    cand_gate = torch.full((T, kc), -7.0, dtype=torch.float32, device=dev)
    rws = torch.zeros(M.route_workspace_size(cfg), dtype=torch.uint8, device=dev)
    M.moe_route(cfg, None, None, None, Ld, scores, None if w.mode == W.EXPERT_CHOICE else cand_idx,
                cand_gate, rws, home_group=cuda(home_group))
    slot = torch.full((T, kc), -7, dtype=torch.int32, device=dev)
    keep = torch.full((T, kc), 7, dtype=torch.uint8, device=dev)
    demand = torch.full((N,), -7, dtype=torch.int32, device=dev)
    kept = torch.full((N,), -7, dtype=torch.int32, device=dev)
    M.moe_capacity_drop(cfg, None if w.mode == W.EXPERT_CHOICE else cand_idx, cand_gate, slot,
                        keep, demand, kept)
    offs = torch.full((N + 1,), -7, dtype=torch.int32, device=dev)
    row_token = torch.full((R,), -7, dtype=torch.int32, device=dev)
    row_gate = torch.full((R,), -7.0, dtype=torch.float32, device=dev)
    tok_rows = torch.full((T, kc), -7, dtype=torch.int32, device=dev)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    xd = cuda(x) if x is not None else torch.zeros((max(T, 1), w.d), dtype=dt, device=dev)
    xp = torch.zeros((R, w.d), dtype=dt, device=dev)
    coverage = torch.full((T,), -7, dtype=torch.int32, device=dev)
    M.moe_dispatch(cfg, xd, None if w.mode == W.EXPERT_CHOICE else cand_idx, cand_gate, slot, kept,
                   offs, row_token, row_gate, tok_rows, xp, coverage=coverage)
    torch.cuda.synchronize()
    out = dict(scores=scores, cand_idx=cand_idx, cand_gate=cand_gate, slot=slot, keep=keep,
               demand=demand, kept=kept, expert_offsets=offs, row_token=row_token,
               row_gate=row_gate, tok_rows=tok_rows, coverage=coverage)
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["xp"] = xp.cpu()
    return res


def compare_routing(w: W.Workload, g: Dict[str, np.ndarray], L: np.ndarray, home_group=None) -> None:
    """Bit-exact comparison of every routing output with the oracle's."""
    rt = oracle_route(w, L, home_group)
    ec = w.mode == W.EXPERT_CHOICE
    assert np.array_equal(g["scores"].view(np.uint32), rt["p"].view(np.uint32)), "scores differ"
    if not ec:
        assert np.array_equal(g["cand_idx"], rt["idx"]), "candidate experts differ"
    assert np.array_equal(g["cand_gate"].view(np.uint32), rt["gate"].view(np.uint32)), "gates differ"
    assert np.array_equal(g["keep"].astype(bool), rt["keep"]), "keep masks differ"
    assert np.array_equal(g["demand"], rt["demand"]), "demand differs"
    assert np.array_equal(g["kept"], rt["kept"]), "kept differs"
    idx = rt["idx"]
    dp = O.dispatch(idx, rt["gate"], rt["keep"], w.N)
    assert np.array_equal(g["slot"], dp["slot"]), "slots differ"
    assert np.array_equal(g["expert_offsets"], dp["expert_offsets"]), "offsets differ"
    P = dp["P"]
    assert np.array_equal(g["row_token"][:P], dp["row_token"]), "row_token differs"
    assert np.array_equal(g["row_gate"][:P].view(np.uint32), dp["row_gate"].view(np.uint32))
    assert np.array_equal(g["tok_rows"], dp["tok_rows"]), "tok_rows differ"
    # coverage from the library, against the oracle's count of experts per token
    assert np.array_equal(g["coverage"], rt["coverage"]), "coverage differs"
    if ec:
        assert int(g["coverage"].sum()) == w.N * O.ec_capacity(w.k, w.T, w.N)


def layer_gpu(w: W.Workload, inp: Dict[str, torch.Tensor], logits: Optional[np.ndarray] = None,
              home_group=None, want_views: bool = False, fuse_gather: bool = False):
    """moe_layer_forward on the GPU. ``logits`` given -> MOE_LOGITS_GIVEN;
    ``fuse_gather`` -> MOE_FUSE_GATHER."""
    cfg = M.config_from_workload(w, logits_given=logits is not None, fuse_gather=fuse_gather)
    dev = torch.device("cuda")
    wsz = M.workspace_size_e4m3(cfg) if w.weights == "e4m3" else M.workspace_size(cfg)
    ws = torch.zeros(wsz, dtype=torch.uint8, device=dev)  # status word = 0
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((w.T, w.d), dtype=dt, device=dev)
    stats = torch.zeros(M.MOE_STATS_LEN, dtype=torch.float64, device=dev)
    Lg = torch.from_numpy(np.ascontiguousarray(logits)).to(dev) if logits is not None else \
        torch.empty((w.T, w.N), dtype=torch.float32, device=dev)
    if w.weights == "e4m3":
        q = {k: cuda(inp[k]) for k in ("W1q", "W3q", "W2q", "W1s", "W3s", "W2s")}
        ex = M.e4m3_experts(q["W1q"], q["W3q"], q["W2q"], q["W1s"], q["W3s"], q["W2s"])
        M.moe_layer_forward_e4m3(cfg, cuda(inp["x"]), cuda(inp["W_r"]), cuda(inp["bias"]), ex,
                                 cuda(inp.get("Ws1")), cuda(inp.get("Ws3")), cuda(inp.get("Ws2")),
                                 y, ws, home_group=cuda(home_group), logits=Lg, stats=stats)
    else:
        M.moe_layer_forward(cfg, cuda(inp["x"]), cuda(inp["W_r"]), cuda(inp["bias"]),
                            cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                            cuda(inp.get("Ws1")), cuda(inp.get("Ws3")), cuda(inp.get("Ws2")), y, ws,
                            home_group=cuda(home_group), logits=Lg, stats=stats)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    out = dict(y=np32(y), logits=Lg.cpu().numpy(), stats=stats.cpu().numpy())
    if want_views:
        v = M.moe_workspace_views(cfg, ws)
        sz = M.sizes(cfg)
        out["kept"] = M.view_tensor(v.kept, (w.N,), torch.int32).cpu().numpy()
        out["keep"] = M.view_tensor(v.keep, (w.T, sz.kc), torch.uint8).cpu().numpy()
        out["cand_idx"] = M.view_tensor(v.cand_idx, (w.T, sz.kc), torch.int32).cpu().numpy()
        out["coverage"] = M.view_tensor(v.coverage, (w.T,), torch.int32).cpu().numpy()
    return out


def oracle_layer(w: W.Workload, inp: Dict[str, torch.Tensor], logits: Optional[np.ndarray] = None,
                 tokens=None, home_group=None):
    if w.weights == "e4m3":  # the experts the GPU multiplies: e4m3 values times column scales
        W1, W3, W2 = (O.dequantize_e4m3(inp[n + "q"].numpy(), inp[n + "s"].numpy(), kmajor=True)
                      for n in ("W1", "W3", "W2"))
    else:
        W1, W3, W2 = np32(inp["W1"]), np32(inp["W3"]), np32(inp["W2"])
    return O.layer_forward(np32(inp["x"]), np32(inp["W_r"]), np32(inp["bias"]), W1,
                           W3, W2, mode=w.mode, k=w.k, gamma=w.gamma,
                           m=w.m, group_size=w.group_size, renorm=w.renorm, dtype=w.dtype,
                           Ws1=np32(inp.get("Ws1")), Ws3=np32(inp.get("Ws3")),
                           Ws2=np32(inp.get("Ws2")), logits=logits, tokens=tokens,
                           home_group=home_group, act_e4m3=w.weights == "e4m3")


def tile_edge_tokens(w: W.Workload, L: np.ndarray, tile: int = 128) -> np.ndarray:
    """Tokens whose rows sit at the first and the last row of every
    ``tile``-row block of every expert segment (the grouped GEMMs tile each
    segment in 128-row blocks, or 256-row blocks split over a CTA pair), and
    at the edges of the shared expert's T-row segment. A token sample that
    contains them exercises every tile, including each segment's ragged last
    tile, at the workload's full K depth."""
    rt = oracle_route(w, L)
    dp = O.dispatch(rt["idx"], rt["gate"], rt["keep"], w.N)
    off, row_token = dp["expert_offsets"], dp["row_token"]
    rows = []
    for e in range(w.N):
        lo, hi = int(off[e]), int(off[e + 1])
        for a in range(lo, hi, tile):
            rows += [a, min(a + tile, hi) - 1]
    toks = set(int(row_token[r]) for r in rows)
    if w.f_shared:
        for a in range(0, w.T, tile):
            toks.update((a, min(a + tile, w.T) - 1))
    return np.array(sorted(toks), dtype=np.int64)


def logit_bound(x: np.ndarray, W_r: np.ndarray, L: np.ndarray) -> np.ndarray:
    """Worst-case fp32 accumulation error of L = x W_r + b (Higham gamma_d):
    d * 2^-24 * sum_j |x_j| |w_je|, plus the roundings of the bias add and of
    the reference itself (2^-23 |L| each)."""
    d = x.shape[1]
    s = np.abs(x.astype(np.float64)) @ np.abs(W_r.astype(np.float64))
    return (d + 2) * 2.0 ** -24 * s + 2.0 ** -22 * np.abs(L.astype(np.float64)) + 1e-30
