"""CPU oracle for one sparse Mixture-of-Experts FFN layer forward pass.

TEST INFRASTRUCTURE. This module exists to check the CUDA library; it is not
part of the product path. Only the test suite, the package smoke check and the
benchmark's CPU-baseline/reference leg may import it. It shares no code with
the CUDA library and imports nothing from it.

It is written as a plain, slow, direct reading of the pages it cites:

* "Understanding Mixture of Experts" (dongbusteel.co.kr), §"How MoE differs
  from the Transformer": the layer output is y = sum_i G(x)_i * E_i(x), with
  E_i an expert network and G(x) the router's selection weights; §"Expert and
  Router": the router activates the TopK(G(x), k) experts of each token.
* "MoE vs MoT: routing and inference cost" (hrletsgo.me), §"MoE basic
  structure": the FFN is replicated N times and each token passes through its
  top-k; §"Mixture of Tokens": expert choice, each expert takes the c = k*T/N
  tokens of the batch with the highest router score, so every expert processes
  exactly c tokens while a token may be taken by several experts or by none;
  §"MoE basic structure" also names the Switch balance term, the sum over
  experts of f_i * P_i.
* "Capacity-Aware Inference: Mitigating the Straggler Effect in MoE"
  (gist.science summary of arXiv 2503.05066), §2① Capacity-Aware Token Drop:
  each expert has capacity C = gamma * N_bar and the tokens beyond it with the
  lowest gating scores are dropped; §2② Capacity-Aware Expanded Drop: a token's
  candidate set grows by m local experts of the same device; §2③
  Device-Level Capacity-Aware Inference: the capacity is held per device, so an
  expert over its own share keeps its tokens while its device has room.
* "How to design inference cost with MoE routing" (blog.gillilab.com),
  §"how routing allocates the compute budget": a shared expert that every token
  passes through.

Readings taken where the pages are silent (each repeated where it is used):
  R1 expert form: SwiGLU, E(x) = (silu(x W1) * (x W3)) W2, no biases.
  R2 G(x) = softmax of router logits (temperature 1, no noise); entries of
     experts a token does not use are 0.
  R3 scores are computed by one fixed fp32 operation sequence (max, subtract,
     a Cody-Waite exponential, left-to-right sum, correctly rounded divide), so
     that every integer decision made from them is reproducible bit for bit.
  R4 ties: top-k prefers the lower expert index; expert choice and capacity drop
     prefer the lower token index. -0.0 ranks equal to +0.0.
  R5 N_bar = k*T/N (mean tokens per expert, using k and not k+m);
     C = floor(gamma * N_bar) in fp64, capped at T; gamma = inf means no limit;
     c = min(T, floor(k*T/N)).
  R6 the gating score that ranks drops is the gate the pair is weighted by
     (after renormalisation when renorm is on); drops are per (token, expert)
     pair and the surviving gates are not renormalised again.
  R7 expanded drop: a token's device is its contiguous shard of the batch,
     group floor(t*G/T) of G = N/group_size groups of consecutive experts,
     unless a home group is given; its m extra candidates are the group's
     highest-logit experts not already in its top-k.
  R8 storage points: bf16 layers keep x, weights, the SwiGLU hidden h, each
     expert output and y in bf16; fp32 layers keep them in fp32; every sum and
     product is taken in fp64 here and rounded only at those points.
  R14 FP8 experts: the routed experts' weights are e4m3 bytes with one fp32
     scale per output column (input preparation); both operands of each
     expert product are e4m3, the activation rows (the token rows before W1
     and W3, the stored hidden rows before W2) quantized per row with scale
     max|row| / 448; products of e4m3 values, fp32 scales applied to the sums.
  R13 device-level capacity: a device is the group of `group_size` consecutive
     experts (as in R7); its capacity is the sum of its experts' capacities,
     floor(gamma * N_bar * group_size), capped at T * min(kc, group_size);
     over capacity the device keeps its highest-gate candidates, ties to the
     lower token, then to the token's earlier candidate slot; tokens are not
     moved between experts.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

F32 = np.float32

# --------------------------------------------------------------------------
# Storage rounding (reading R8)
# --------------------------------------------------------------------------


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as fp32.

    Works on the fp64 value so it is rounded once, not twice. bf16 has the
    exponent range of fp32 and 8 significant bits: a normal magnitude (at
    least 2**-126) keeps the top 8 bits of its significand; below 2**-126 the
    bf16 values are the subnormals m * 2**-133 (m = 0..127), so the value is
    rounded to the nearest multiple of 2**-133, ties to even m (m = 128 is
    the smallest normal, 2**-126).
    """
    a = np.asarray(v, dtype=np.float64)
    bits = a.view(np.uint64)
    # bf16 keeps 8 significant bits; fp64 has 53: drop the low 45 bits, RNE.
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    rounded = (bits + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    out = rounded.view(np.float64)
    # a * 2**133 is exact in fp64 and np.rint rounds half to even
    sub = np.rint(a * 2.0 ** 133) * 2.0 ** -133
    out = np.where(np.abs(a) < 2.0 ** -126, sub, out)
    return out.astype(np.float32)


def store(v, dtype: str) -> np.ndarray:
    """Round a fp64 result at a storage point of the layer (reading R8)."""
    if dtype == "bf16":
        return round_bf16(v).astype(np.float64)
    if dtype == "f32":
        return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(v, dtype=np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# Router logits and scores (readings R2, R3)
# --------------------------------------------------------------------------


def router_logits(x, W_r, bias=None) -> np.ndarray:
    """L[t, e] = sum_j x[t, j] * W_r[j, e] + b_e in fp64, rounded once to fp32.

    The router scores every token against every expert ("Understanding Mixture
    of Experts", §"Expert and Router").
    """
    L = np.asarray(x, np.float64) @ np.asarray(W_r, np.float64)
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L.astype(F32)


# Cody-Waite range reduction (W. J. Cody and W. Waite, "Software Manual for
# the Elementary Functions", 1980) followed by the degree-7 Taylor polynomial
# of exp on |r| <= ln2/2, all in fp32 with round-to-nearest-even.
#   LN2_HI: ln 2 truncated to 16 significant bits, so n*LN2_HI is exact in
#           fp32 for |n| < 2**8 and x - n*LN2_HI is exact (Sterbenz).
#   LN2_LO: ln 2 - LN2_HI rounded to fp32.
LOG2E = F32(1.0 / math.log(2.0))
LN2_HI = F32(math.floor(math.log(2.0) * 2.0 ** 16) / 2.0 ** 16)
LN2_LO = F32(math.log(2.0) - float(LN2_HI))
TAYLOR = [F32(1.0 / math.factorial(i)) for i in range(8)]


def rexp(x) -> np.ndarray:
    """exp(x) for fp32 x <= 0 by the fixed fp32 sequence of reading R3.

    n = rint(x * LOG2E); r = (x - n*LN2_HI) - n*LN2_LO;
    q = Horner(1/7!, ..., 1/1!, 1/0!) in r with separate multiply and add;
    result = q * 2**n, or 0 when n < -125.
    """
    x = np.asarray(x, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore"):
        return _rexp(x)


def _rexp(x):
    n = np.rint(x * LOG2E).astype(F32)          # fp32 multiply, ties-to-even
    r = (x - n * LN2_HI).astype(F32)
    r = (r - n * LN2_LO).astype(F32)
    q = TAYLOR[7]
    for i in range(6, -1, -1):
        q = (q * r).astype(F32)
        q = (q + TAYLOR[i]).astype(F32)
    q = np.broadcast_to(q, x.shape).astype(F32)
    big = n < F32(-125.0)
    n_int = np.where(big, 0, n).astype(np.int32)
    out = np.ldexp(q, n_int).astype(F32)
    return np.where(big, F32(0.0), out).astype(F32)


def softmax_scores(L) -> np.ndarray:
    """p[t, e] = G(x_t)_e, the softmax of the logits over experts (reading R2),
    by the fp32 sequence of reading R3:
        m_t = max_e L[t, e];  u_e = rexp(L[t, e] - m_t);
        Z_t = (((u_0 + u_1) + u_2) + ...);  p[t, e] = u_e / Z_t.
    """
    L = np.asarray(L, dtype=F32)
    T, N = L.shape
    m = L.max(axis=1, keepdims=True)
    u = rexp((L - m).astype(F32))
    Z = u[:, 0].copy()
    for e in range(1, N):
        Z = (Z + u[:, e]).astype(F32)
    return (u / Z[:, None]).astype(F32)


# --------------------------------------------------------------------------
# Ordering keys (reading R4)
# --------------------------------------------------------------------------


def key32(v) -> np.ndarray:
    """Unsigned 32-bit key that orders finite fp32 values like the values
    themselves, with -0.0 mapped to the key of +0.0."""
    v = np.asarray(v, dtype=F32)
    v = np.where(v == F32(0.0), F32(0.0), v).astype(F32)
    u = v.view(np.uint32)
    neg = (u >> np.uint32(31)) == 1
    return np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


# --------------------------------------------------------------------------
# Token choice, expanded candidates, gates
# --------------------------------------------------------------------------


def topk_experts(L, k: int) -> np.ndarray:
    """idx[t, 0..k-1]: the k experts with the largest logits of token t, best
    first, ties to the lower expert index (TopK(G(x), k) of "Understanding
    Mixture of Experts", §"Expert and Router"; reading R4). Softmax is
    monotone, so ranking logits ranks G(x)."""
    keys = key32(L).astype(np.int64)
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def home_groups(T: int, n_groups: int) -> np.ndarray:
    """Reading R7: token t lives on device floor(t * G / T)."""
    return (np.arange(T, dtype=np.int64) * n_groups // T).astype(np.int32)


def expanded_candidates(L, idx, m: int, group_size: int, home_group=None) -> np.ndarray:
    """Append m extra candidates per token from the experts of its own device
    ("Capacity-Aware Inference", §2② Expanded Drop; reading R7).

    Returns idx_ext[T, k+m]; slots with no candidate left hold -1."""
    L = np.asarray(L, dtype=F32)
    T, N = L.shape
    k = idx.shape[1]
    G = N // group_size
    hg = home_groups(T, G) if home_group is None else np.asarray(home_group)
    out = np.full((T, k + m), -1, dtype=np.int32)
    out[:, :k] = idx
    for t in range(T):
        g = int(hg[t])
        members = [e for e in range(g * group_size, (g + 1) * group_size)
                   if e not in set(idx[t].tolist())]
        members.sort(key=lambda e: (-int(key32(L[t, e])), e))
        for j, e in enumerate(members[:m]):
            out[t, k + j] = e
    return out


def token_gates(p, idx, renorm: bool) -> np.ndarray:
    """gate[t, j] = p[t, idx[t, j]] (0 for an empty slot). With renorm the
    gates of a token are divided by their fp32 sum taken left to right in slot
    order (reading R6)."""
    p = np.asarray(p, dtype=F32)
    T, kc = idx.shape
    g = np.zeros((T, kc), dtype=F32)
    valid = idx >= 0
    rows = np.repeat(np.arange(T)[:, None], kc, axis=1)
    g[valid] = p[rows[valid], idx[valid]]
    if renorm:
        S = g[:, 0].copy()
        for j in range(1, kc):
            S = (S + g[:, j]).astype(F32)
        g = (g / S[:, None]).astype(F32)
    return g


# --------------------------------------------------------------------------
# Capacity drop and expert choice
# --------------------------------------------------------------------------


def capacity(gamma: float, k: int, T: int, N: int) -> int:
    """C = floor(gamma * N_bar), N_bar = k*T/N, in fp64, capped at T; gamma =
    inf means no limit ("Capacity-Aware Inference", §2①; reading R5)."""
    if math.isinf(gamma):
        return T
    nbar = (k * T) / N
    return int(min(math.floor(gamma * nbar), T))


def ec_capacity(k: int, T: int, N: int) -> int:
    """c = k*T/N tokens per expert ("MoE vs MoT", §"Mixture of Tokens";
    reading R5)."""
    return min(T, (k * T) // N)


def capacity_drop(idx, gate, N: int, C: int):
    """Per expert, keep at most C of its candidates: the ones with the highest
    gating score, ties to the lower token; drop the rest ("Capacity-Aware
    Inference", §2① Token Drop; readings R4, R6).

    Returns keep[T, kc] (bool), demand[N] (candidates before the drop) and
    kept[N] (after)."""
    idx = np.asarray(idx)
    T, kc = idx.shape
    keep = np.zeros((T, kc), dtype=bool)
    demand = np.zeros(N, dtype=np.int64)
    kept = np.zeros(N, dtype=np.int64)
    gk = key32(gate).astype(np.int64)
    for e in range(N):
        ts, js = np.nonzero(idx == e)
        demand[e] = len(ts)
        if len(ts) <= C:
            sel = np.arange(len(ts))
        else:
            order = np.lexsort((ts, -gk[ts, js]))     # key desc, then token asc
            sel = order[:C]
        keep[ts[sel], js[sel]] = True
        kept[e] = len(sel)
    return keep, demand, kept


def device_capacity(gamma: float, k: int, T: int, N: int, group_size: int, kc: int) -> int:
    """Capacity of one device, a group of `group_size` experts, for
    device-level capacity-aware inference ("Capacity-Aware Inference", §2③:
    capacity is managed per device instead of per expert; reading R13): the
    sum of its experts' capacities, floor(gamma * N_bar * group_size) in fp64
    with N_bar = k*T/N, capped at the largest possible device demand
    T * min(kc, group_size); gamma = inf means no limit."""
    most = T * min(kc, group_size)
    if math.isinf(gamma):
        return most
    nbar = (k * T) / N
    return int(min(math.floor(gamma * nbar * group_size), most))


def device_capacity_drop(idx, gate, N: int, group_size: int, C_dev: int):
    """Device-level capacity-aware drop ("Capacity-Aware Inference", §2③;
    reading R13): the candidates of all experts of a device (a group of
    `group_size` consecutive experts) share one capacity C_dev; an expert may
    exceed its own share as long as the device has room. Over capacity, the
    device keeps the C_dev candidates with the highest gating score, ties to
    the lower token and then to the token's earlier candidate slot.

    Returns keep[T, kc] (bool), demand[N] and kept[N] per expert."""
    idx = np.asarray(idx)
    T, kc = idx.shape
    keep = np.zeros((T, kc), dtype=bool)
    gk = key32(gate).astype(np.int64)
    for lo in range(0, N, group_size):
        ts, js = np.nonzero((idx >= lo) & (idx < lo + group_size))
        if len(ts) <= C_dev:
            sel = np.arange(len(ts))
        else:
            order = np.lexsort((js, ts, -gk[ts, js]))   # key desc, token asc, slot asc
            sel = order[:C_dev]
        keep[ts[sel], js[sel]] = True
    demand = np.array([(idx == e).sum() for e in range(N)], dtype=np.int64)
    kept = np.array([((idx == e) & keep).sum() for e in range(N)], dtype=np.int64)
    return keep, demand, kept


def expert_choice(p, c: int):
    """Each expert takes the c tokens with the highest score p[:, e], ties to
    the lower token ("MoE vs MoT", §"Mixture of Tokens"; reading R4).

    Returns keep[T, N] (bool; column e marks expert e's tokens) and coverage[T],
    the number of experts that took each token."""
    p = np.asarray(p, dtype=F32)
    T, N = p.shape
    keep = np.zeros((T, N), dtype=bool)
    keys = key32(p).astype(np.int64)
    tok = np.arange(T)
    for e in range(N):
        order = np.lexsort((tok, -keys[:, e]))
        keep[order[:c], e] = True
    return keep, keep.sum(axis=1).astype(np.int64)


# --------------------------------------------------------------------------
# Routing as a whole
# --------------------------------------------------------------------------


def route(L, *, mode: str, k: int, N: int, gamma: float = math.inf, m: int = 0,
          group_size: int = 8, renorm: bool = False, home_group=None) -> Dict[str, np.ndarray]:
    """All routing decisions of one batch from its fp32 logits.

    Returns a dict with:
      p        [T, N] fp32 scores
      idx      [T, kc] expert of each candidate slot (-1 = empty); expert
               choice uses kc = N and idx[t, j] = j
      gate     [T, kc] fp32 gate of each slot
      keep     [T, kc] bool, slot survives selection
      demand   [N] candidates per expert before selection
      kept     [N] pairs per expert after selection
      coverage [T] kept pairs per token
      C        capacity in force (T when unlimited; c for expert choice)
    """
    L = np.asarray(L, dtype=F32)
    T = L.shape[0]
    p = softmax_scores(L)
    if mode == "expert_choice":
        c = ec_capacity(k, T, N)
        keep, coverage = expert_choice(p, c)
        idx = np.broadcast_to(np.arange(N, dtype=np.int32), (T, N)).copy()
        gate = p.copy()
        kept = keep.sum(axis=0).astype(np.int64)
        return dict(p=p, idx=idx, gate=gate, keep=keep, demand=kept.copy(), kept=kept,
                    coverage=coverage, C=c)
    idx = topk_experts(L, k)
    if m > 0:
        idx = expanded_candidates(L, idx, m, group_size, home_group)
    gate = token_gates(p, idx, renorm)
    if mode == "capacity_drop_device":
        C = device_capacity(gamma, k, T, N, group_size, idx.shape[1])
        keep, demand, kept = device_capacity_drop(idx, gate, N, group_size, C)
        return dict(p=p, idx=idx, gate=gate, keep=keep, demand=demand, kept=kept,
                    coverage=keep.sum(axis=1).astype(np.int64), C=C)
    C = capacity(gamma, k, T, N) if mode == "capacity_drop" else T
    keep, demand, kept = capacity_drop(idx, gate, N, C)
    return dict(p=p, idx=idx, gate=gate, keep=keep, demand=demand, kept=kept,
                coverage=keep.sum(axis=1).astype(np.int64), C=C)


def dispatch(idx, gate, keep, N: int) -> Dict[str, np.ndarray]:
    """Expert-contiguous row order of the kept pairs.

    expert_offsets[e] = sum of kept pairs of experts < e; inside an expert the
    rows follow ascending token; tok_rows[t] lists token t's rows in ascending
    expert order (equivalently ascending row), padded with -1; slot[t, j] is the
    row of candidate (t, j) relative to its expert's first row, or -1.
    """
    idx = np.asarray(idx)
    T, kc = idx.shape
    kept = np.array([int(np.sum(keep & (idx == e))) for e in range(N)], dtype=np.int64)
    offsets = np.zeros(N + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    P = int(offsets[-1])
    row_token = np.zeros(P, dtype=np.int64)
    row_gate = np.zeros(P, dtype=F32)
    slot = np.full((T, kc), -1, dtype=np.int64)
    for e in range(N):
        ts, js = np.nonzero(keep & (idx == e))        # row-major: ascending t
        r = offsets[e] + np.arange(len(ts))
        row_token[r] = ts
        row_gate[r] = gate[ts, js]
        slot[ts, js] = np.arange(len(ts))
    tok_rows = np.full((T, kc), -1, dtype=np.int64)
    for t in range(T):
        rows = sorted(int(offsets[idx[t, j]] + slot[t, j]) for j in range(kc) if keep[t, j])
        tok_rows[t, :len(rows)] = rows
    return dict(expert_offsets=offsets, row_token=row_token, row_gate=row_gate,
                slot=slot, tok_rows=tok_rows, P=P)


# --------------------------------------------------------------------------
# Experts and combine (readings R1, R8)
# --------------------------------------------------------------------------


def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(X, W1e, W3e, W2e, dtype: str, act_e4m3: bool = False) -> np.ndarray:
    """E(X) = (silu(X W1) * (X W3)) W2 in fp64, rounding h and the result at
    the layer's storage points (readings R1, R8).

    ``act_e4m3`` (reading R14, experts in FP8): the operand rows of both
    products are quantized to e4m3 first, X before W1 and W3, the stored h
    before W2 (quantize_rows_e4m3), and the products use their dequantized
    values, exactly in fp64."""
    X = np.asarray(X, np.float64)
    if act_e4m3:
        X = dequantize_rows_e4m3(*quantize_rows_e4m3(X))
    a = X @ np.asarray(W1e, np.float64)
    g = X @ np.asarray(W3e, np.float64)
    h = store(silu(a) * g, dtype)
    if act_e4m3:
        h = dequantize_rows_e4m3(*quantize_rows_e4m3(h))
    return store(h @ np.asarray(W2e, np.float64), dtype)


def layer_forward(x, W_r, bias, W1, W3, W2, *, mode: str, k: int, gamma: float = math.inf,
                  m: int = 0, group_size: int = 8, renorm: bool = False, dtype: str = "bf16",
                  Ws1=None, Ws3=None, Ws2=None, logits=None, home_group=None,
                  tokens=None, act_e4m3: bool = False) -> Dict[str, np.ndarray]:
    """y_t = sum over kept pairs (t, e), in ascending e, of gate * E_e(x_t),
    plus the shared expert's output when one is given; a token with no kept
    pair and no shared expert outputs 0 ("Understanding Mixture of Experts",
    layer equation; "How to design inference cost with MoE routing", shared
    expert).

    ``logits`` replaces the router GEMM with given fp32 logits. ``tokens``
    computes the output rows of those tokens only (routing is always computed
    for the whole batch, since capacity and expert choice couple all tokens);
    y then has one row per listed token. ``act_e4m3``: the routed experts run
    in FP8 (reading R14: their weights are given dequantized, their operand
    rows are quantized to e4m3 per row); the shared expert is unchanged.
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    N = W1.shape[0]
    L = router_logits(x, W_r, bias) if logits is None else np.asarray(logits, dtype=F32)
    rt = route(L, mode=mode, k=k, N=N, gamma=gamma, m=m, group_size=group_size,
               renorm=renorm, home_group=home_group)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    pos = {int(t): i for i, t in enumerate(tok)}
    acc = np.zeros((len(tok), x.shape[1]), dtype=np.float64)
    idx, gate, keep = rt["idx"], rt["gate"], rt["keep"]
    for e in range(N):
        ts, js = np.nonzero(keep & (idx == e))
        sel = [i for i, t in enumerate(ts) if int(t) in pos]
        if not sel:
            continue
        ts, js = ts[sel], js[sel]
        o = swiglu(x[ts], W1[e], W3[e], W2[e], dtype, act_e4m3=act_e4m3)
        rows = np.array([pos[int(t)] for t in ts])
        acc[rows] += gate[ts, js].astype(np.float64)[:, None] * o
    if Ws1 is not None:
        acc += swiglu(x[tok], Ws1, Ws3, Ws2, dtype)
    rt["logits"] = L
    rt["y"] = store(acc, dtype)
    rt["tokens"] = tok
    return rt


# --------------------------------------------------------------------------
# FP8 expert weights
# --------------------------------------------------------------------------


def e4m3_value(b) -> np.ndarray:
    """Values of e4m3 bytes (1 sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; exponent 0 holds the subnormals m * 2^-9; the byte pattern
    with all exponent and mantissa bits set is NaN; there is no infinity)."""
    b = np.asarray(b, dtype=np.int64)
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return np.where(s == 1, -val, val)


def dequantize_e4m3(q, scale, kmajor: bool = False) -> np.ndarray:
    """Expert weights stored as e4m3 bytes q [..., K, n] (or, with kmajor,
    [..., n, K]: each output column's K bytes contiguous) with one fp32 scale
    per output column, scale [..., n]: W[k, n] = value(q) * scale[n], exact in
    fp64, returned as [..., K, n]."""
    v = e4m3_value(q)
    if kmajor:
        v = np.swapaxes(v, -1, -2)
    return v * np.asarray(scale, np.float64)[..., None, :]


E4M3_MAX = 448.0  # largest finite e4m3 magnitude, 1.75 * 2^8


def round_e4m3(v) -> np.ndarray:
    """The e4m3 value nearest to each v (fp64), ties to the even code, finite
    magnitudes beyond 448 saturated to 448; the sign is kept (also on zero).

    e4m3 values: in the binade [2^e, 2^(e+1)), e >= -6, the step is 2^(e-3)
    (3 mantissa bits); below 2^-6 the subnormals m * 2^-9. Rounding a/step to
    the nearest integer, ties to even, is ties-to-even of the code's last
    mantissa bit."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))     # a = m * 2^ex, 0.5 <= m < 1
    e = np.maximum(ex - 1, -6)
    step = np.ldexp(1.0, e - 3)
    r = np.rint(a / step) * step                  # a / step: exact (a power-of-two scaling)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def quantize_rows_e4m3(X):
    """One fp32 scale per row and e4m3 values (reading R14, activations of the
    FP8 experts): amax = max |X[r, :]| (exact), scale = amax / 448 rounded to
    fp32 (1 for an all-zero row), v = X / scale rounded to fp32 (correctly
    rounded division), then the nearest e4m3 value of v (round_e4m3).

    Returns (values [R, K] fp64, each an e4m3 value; scale [R] fp32)."""
    Xf = np.asarray(X, np.float64).astype(np.float32)
    if Xf.ndim != 2:
        raise ValueError("rows of a matrix")
    amax = np.max(np.abs(Xf), axis=1) if Xf.shape[1] else np.zeros(Xf.shape[0], F32)
    scale = np.where(amax > 0, (amax / F32(E4M3_MAX)).astype(F32), F32(1.0)).astype(F32)
    v = (Xf / scale[:, None]).astype(F32)
    return round_e4m3(v.astype(np.float64)), scale


def dequantize_rows_e4m3(values, scale) -> np.ndarray:
    """Row r of the quantized matrix times its scale, exact in fp64."""
    return np.asarray(values, np.float64) * np.asarray(scale, np.float64)[:, None]


# --------------------------------------------------------------------------
# Load statistics
# --------------------------------------------------------------------------


def load_stats(demand, kept, p) -> Dict[str, float]:
    """Switch balance term B = sum_i f_i * P_i ("MoE vs MoT", §"MoE basic
    structure") with f_i = demand_i / sum(demand) (candidates before any drop)
    and P_i = mean_t p[t, i]; N*B is 1 for a perfectly even router. Also the
    straggler indicator max/mean kept load ("Capacity-Aware Inference", §1) and
    the dropped fraction of candidate pairs."""
    demand = np.asarray(demand, np.float64)
    kept = np.asarray(kept, np.float64)
    p = np.asarray(p, np.float64)
    N = demand.shape[0]
    f = demand / demand.sum() if demand.sum() > 0 else np.zeros(N)
    P = p.sum(axis=0) / p.shape[0]
    B = float(np.sum(f * P))
    mean = kept.mean()
    return dict(P=float(kept.sum()), demand_total=float(demand.sum()),
                max_kept=float(kept.max()), mean_kept=float(mean),
                max_over_mean=float(kept.max() / mean) if mean > 0 else 0.0,
                drop_fraction=float(1.0 - kept.sum() / demand.sum()) if demand.sum() > 0 else 0.0,
                balance=B, balance_times_N=N * B)
