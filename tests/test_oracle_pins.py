"""Pins of the CPU oracle to facts outside itself: hand-worked examples,
closed forms, library routines, brute force on tiny inputs and invariants the
pages state. A plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a wrong tie-break) fails at least one of these."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_workloads as W
import oracle as O

F32 = np.float32


def _gamma(v):
    return math.inf if v == "inf" else float(v)


# ---------------------------------------------------------------- exp and keys

def test_cody_waite_constants_from_ln2():
    ln2 = math.log(2.0)
    hi = float(O.LN2_HI)
    # at most 16 significant bits, so n*hi is exact in fp32 for |n| < 2**8
    assert hi * 2 ** 16 == math.floor(hi * 2 ** 16)
    assert abs(hi - ln2) < 2.0 ** -16
    assert abs(hi + float(O.LN2_LO) - ln2) < 2.0 ** -40
    assert O.LOG2E == F32(1.0 / ln2)
    for i, c in enumerate(O.TAYLOR):
        assert c == F32(1.0 / math.factorial(i))


def test_rexp_against_libm_within_two_ulp():
    x = np.concatenate([np.linspace(-87.0, 0.0, 400001, dtype=F32),
                        -np.abs(np.random.default_rng(1).standard_normal(100000)).astype(F32) * 4])
    got = O.rexp(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(F32)).astype(np.float64)
    normal = ref >= 2.0 ** -124
    assert np.max(np.abs(got - ref)[normal] / ulp[normal]) <= 2.0
    # below that the sequence flushes to zero, and only there
    assert np.all(got[~normal & (got == 0)] == 0) and np.all(ref[got == 0] < 2.0 ** -124)
    assert O.rexp(np.array([0.0], F32))[0] == F32(1.0)
    assert O.rexp(np.array([-200.0, -1e30], F32)).tolist() == [0.0, 0.0]


def test_key32_orders_like_values():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.standard_normal(2000).astype(F32) * 10,
                        np.array([0.0, -0.0, 1e-45, -1e-45, 3e38, -3e38, 1.0, -1.0], F32)])
    k = O.key32(v)
    for a, b in itertools.product(range(0, len(v), 37), range(0, len(v), 41)):
        assert (v[a] < v[b]) == (k[a] < k[b])
        assert (v[a] == v[b]) == (k[a] == k[b])
    assert O.key32(np.array([-0.0], F32))[0] == O.key32(np.array([0.0], F32))[0]


def test_round_bf16_matches_torch_and_rounds_once():
    v = np.random.default_rng(3).standard_normal(100000).astype(F32) * 7
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(O.round_bf16(v), ref)
    # 1 + 2**-8 + 2**-30 lies just above the bf16 midpoint 1 + 2**-8: a single
    # rounding goes up, rounding through fp32 first would tie to 1.0
    assert O.round_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == F32(1.0078125)
    assert O.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == F32(1.0)


def test_round_bf16_subnormals_round_to_nearest_even():
    # bf16 subnormals are m * 2**-133, m = 1..127; the rounding keeps them
    # (round to nearest, ties to even m) instead of flushing to zero
    q = 2.0 ** -133
    cases = [(0.5 * q, 0.0), (0.75 * q, q), (1.5 * q, 2 * q), (2.5 * q, 2 * q), (3.5 * q, 4 * q),
             (-1.25 * q, -q), (127.5 * q, 128 * q), (2.0 ** -126 - 2.0 ** -140, 2.0 ** -126),
             (2.0 ** -126, 2.0 ** -126), (1e-45, 0.0)]
    got = O.round_bf16(np.array([a for a, _ in cases]))
    assert got.tolist() == [F32(b) for _, b in cases]
    # a single rounding from fp64: just above a subnormal midpoint goes up
    assert O.round_bf16(np.array([0.5 * q + 2.0 ** -170]))[0] == F32(q)
    # against torch's fp32 -> bf16 conversion over the whole subnormal range
    # and across the boundary 2**-126
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.uniform(-2.0 ** -126, 2.0 ** -126, 50000),
                        rng.uniform(2.0 ** -127, 2.0 ** -125, 20000),
                        np.arange(-300, 300) * 2.0 ** -135]).astype(F32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(O.round_bf16(v), ref)
    assert np.count_nonzero(ref[np.abs(v) < 2.0 ** -126]) > 40000


# ------------------------------------------------------------ softmax / logits

def test_router_logits_closed_form():
    # identity rows of x pick out rows of W_r, plus the bias
    W_r = np.arange(12, dtype=F32).reshape(3, 4) / 7
    b = np.array([0.5, -1.0, 0.0, 2.0], F32)
    L = O.router_logits(np.eye(3, dtype=F32), W_r, b)
    assert np.array_equal(L, (W_r.astype(np.float64) + b).astype(F32))


def test_softmax_scores_against_fp64_and_sum():
    L = W.random_logits(512, 64, seed=4, scale=3.0).numpy()
    p = O.softmax_scores(L)
    Lf = L.astype(np.float64)
    ref = np.exp(Lf - Lf.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    rel = np.abs(p - ref) / np.maximum(ref, 1e-30)
    assert rel[ref > 1e-30].max() < 64 * 2.0 ** -24
    assert np.abs(p.astype(np.float64).sum(1) - 1).max() <= 64 * 2.0 ** -24
    # uniform logits: every expert gets exactly 1/N for N a power of two
    assert np.all(O.softmax_scores(np.zeros((3, 8), F32)) == F32(0.125))


# --------------------------------------------------------------- token choice

def _brute_topk(row, k):
    return sorted(range(len(row)), key=lambda e: (-float(row[e]), e))[:k]


@pytest.mark.parametrize("quantum", [None, 0.5])
def test_topk_brute_force(quantum):
    L = W.random_logits(300, 8, seed=5, quantum=quantum).numpy()
    idx = O.topk_experts(L, 3)
    for t in range(L.shape[0]):
        assert idx[t].tolist() == _brute_topk(L[t], 3)


def test_topk_k_equals_N_and_negative_zero():
    L = np.array([[0.0, -0.0, 1.0, -0.0]], F32)
    assert O.topk_experts(L, 4)[0].tolist() == [2, 0, 1, 3]


def test_renormalised_gates_sum_to_one():
    L = W.random_logits(200, 16, seed=6, scale=2).numpy()
    p = O.softmax_scores(L)
    idx = O.topk_experts(L, 4)
    g = O.token_gates(p, idx, renorm=True)
    assert np.abs(g.astype(np.float64).sum(1) - 1).max() <= 8 * 2.0 ** -24
    graw = O.token_gates(p, idx, renorm=False)
    assert np.array_equal(graw, np.take_along_axis(p, idx.astype(np.int64), 1))


# ------------------------------------------------------- capacity and selection

def test_capacity_values_of_the_workloads():
    assert O.capacity(1.0, 2, 4096, 8) == 1024
    assert O.capacity(1.5, 2, 4096, 8) == 1536
    assert O.capacity(1.25, 6, 8192, 64) == 960
    assert O.capacity(math.inf, 2, 4096, 8) == 4096
    assert O.capacity(1e9, 2, 16, 8) == 16
    assert O.ec_capacity(2, 2048, 16) == 256


def _brute_keep(cands, C):
    """cands: list of (token, gate). The kept set is the unique C-subset whose
    members all rank above every non-member, rank = (gate desc, token asc)."""
    if len(cands) <= C:
        return set(t for t, _ in cands)
    best = None
    for sub in itertools.combinations(range(len(cands)), C):
        inside = [cands[i] for i in sub]
        outside = [cands[i] for i in range(len(cands)) if i not in sub]
        ok = all((a[1] > b[1]) or (a[1] == b[1] and a[0] < b[0])
                 for a in inside for b in outside)
        if ok:
            assert best is None
            best = set(t for t, _ in inside)
    return best


@pytest.mark.parametrize("seed", range(4))
def test_capacity_drop_brute_force_and_invariants(seed):
    T, N, k = 12, 4, 2
    L = W.random_logits(T, N, seed=10 + seed, quantum=0.5).numpy()
    rt = O.route(L, mode="capacity_drop", k=k, N=N, gamma=1.0)
    C = rt["C"]
    assert C == 6
    for e in range(N):
        ts, js = np.nonzero(rt["idx"] == e)
        cands = [(int(t), float(rt["gate"][t, j])) for t, j in zip(ts, js)]
        kept_t = set(int(t) for t, j in zip(ts, js) if rt["keep"][t, j])
        assert kept_t == _brute_keep(cands, C)
        assert rt["kept"][e] == min(rt["demand"][e], C)
    assert rt["kept"].sum() == rt["keep"].sum()


def test_capacity_drop_tight_invariants_larger():
    T, N, k = 2000, 8, 2
    L = W.random_logits(T, N, seed=21, quantum=0.25).numpy()
    L[:, 0] += 1.5                                      # overload expert 0
    rt = O.route(L, mode="capacity_drop", k=k, N=N, gamma=1.0, renorm=True)
    C = rt["C"]
    gk = O.key32(rt["gate"]).astype(np.int64)
    for e in range(N):
        ts, js = np.nonzero(rt["idx"] == e)
        kp = rt["keep"][ts, js]
        assert kp.sum() == min(len(ts), C)
        if (~kp).any() and kp.any():
            kk, dk = gk[ts[kp], js[kp]], gk[ts[~kp], js[~kp]]
            assert kk.min() >= dk.max()
            # at the threshold key, kept tokens precede dropped ones
            thr = kk.min()
            if (dk == thr).any():
                assert ts[kp][kk == thr].max() < ts[~kp][dk == thr].min()
    assert rt["kept"][0] == C and rt["demand"][0] > C


def test_gamma_inf_equals_token_choice_and_zero_drops_all():
    L = W.random_logits(100, 8, seed=7).numpy()
    a = O.route(L, mode="capacity_drop", k=2, N=8, gamma=math.inf)
    b = O.route(L, mode="token_choice", k=2, N=8)
    for key in ("idx", "gate", "keep", "kept", "demand"):
        assert np.array_equal(a[key], b[key])
    assert b["keep"].all()
    z = O.route(L, mode="capacity_drop", k=2, N=8, gamma=0.0)
    assert not z["keep"].any()



# ---------------------------------------------------------- FP8 expert weights

def test_e4m3_values_match_torch_and_hand_values():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).double().numpy()
    got = O.e4m3_value(b)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert O.e4m3_value([0x38, 0x7E, 0x01, 0x08, 0x80, 0xB8])[[0, 1, 2, 3, 5]].tolist() == \
        [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0]
    assert np.signbit(O.e4m3_value([0x80]))[0]


def test_e4m3_quantizer_error_bound_and_dequantization():
    g = torch.Generator().manual_seed(4)
    Wt = (torch.randn(3, 64, 40, generator=g) * 0.05).to(torch.bfloat16)
    Wt[1, :, 7] = 0                                     # an all-zero column
    q, s = W.quantize_e4m3(Wt)
    assert q.dtype == torch.uint8 and s.shape == (3, 40)
    deq = O.dequantize_e4m3(q.numpy(), s.numpy())
    Wd = Wt.double().numpy()
    # each column's largest magnitude maps to 448 * scale, exact up to the scale's rounding
    amax = np.abs(Wd).max(axis=1)
    assert np.allclose(np.abs(deq).max(axis=1), amax, rtol=2 ** -20)
    # round to nearest with 3 mantissa bits: relative error <= 2^-4 above the subnormal range
    big = np.abs(Wd) >= 2.0 ** -6 * s.numpy()[:, None, :]
    assert np.all(np.abs(deq - Wd)[big] <= 2.0 ** -4 * np.abs(Wd)[big] * (1 + 1e-6))
    assert np.all(deq[1, :, 7] == 0)


def _e4m3_table():
    """Every finite e4m3 value with its code (NaN codes left out)."""
    codes = np.arange(256)
    vals = O.e4m3_value(codes)
    ok = ~np.isnan(vals)
    return vals[ok], codes[ok]


def test_round_e4m3_is_the_nearest_code_by_brute_force():
    vals, codes = _e4m3_table()
    rng = np.random.default_rng(41)
    v = np.concatenate([rng.uniform(-470, 470, 3000), rng.uniform(-0.05, 0.05, 3000),
                        rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),
                        (vals[:, None] + vals[None, :]).ravel()[::7] / 2,   # midpoints: ties
                        np.array([0.0, -0.0, 448.0, -448.0, 460.0, 1e6, -1e6])])
    got = O.round_e4m3(v)
    for x, g in zip(v, got):
        if abs(x) > 448:
            assert g == math.copysign(448.0, x)
            continue
        dist = np.abs(vals - x)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:  # a tie: the code whose last mantissa bit is 0
            best = [b for b in best if codes[b] % 2 == 0 and np.signbit(vals[b]) == np.signbit(x)] \
                or [b for b in best if codes[b] % 2 == 0]
        assert g == vals[best[0]], (x, g, vals[best])


def test_round_e4m3_matches_torch_float8():
    rng = np.random.default_rng(42)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(20000) * 2.0 ** -7,
                        rng.uniform(-448, 448, 10000)]).astype(F32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).double().numpy()
    got = O.round_e4m3(v.astype(np.float64))
    fin = np.abs(v) <= 448
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.abs(got[~fin]) == 448.0)


def test_quantize_rows_e4m3_hand_values_and_bounds():
    # a row whose largest magnitude is 448 * 2^-3: the scale is exactly 2^-3 and
    # every e4m3-representable entry comes back unchanged
    q = 2.0 ** -3
    row = np.array([448 * q, -1.5 * q, 0.75 * q, 2.0 ** -9 * q, 0.0])
    vals, scale = O.quantize_rows_e4m3(row[None, :])
    assert scale.dtype == np.float32 and scale[0] == F32(q)
    assert np.array_equal(O.dequantize_rows_e4m3(vals, scale)[0], row)
    # an all-zero row keeps scale 1; the largest magnitude maps to +-448
    vals, scale = O.quantize_rows_e4m3(np.array([[0.0, 0.0], [3.0, -7.0]]))
    assert scale[0] == 1.0 and np.all(vals[0] == 0)
    assert scale[1] == F32(F32(7.0) / F32(448.0)) and vals[1, 1] == -448.0
    # rounding to 3 mantissa bits: relative error <= 2^-4 above the subnormal
    # range of the scaled values, absolute <= 2^-10 * scale below it
    rng = np.random.default_rng(43)
    X = (rng.standard_normal((64, 300)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(F32)
    vals, scale = O.quantize_rows_e4m3(X)
    deq = O.dequantize_rows_e4m3(vals, scale)
    Xd = X.astype(np.float64)
    s = scale.astype(np.float64)[:, None]
    big = np.abs(Xd) >= 2.0 ** -6 * s
    assert np.all(np.abs(deq - Xd)[big] <= 2.0 ** -4 * np.abs(Xd)[big] * (1 + 1e-6))
    assert np.all(np.abs(deq - Xd)[~big] <= 2.0 ** -10 * np.broadcast_to(s, X.shape)[~big] * (1 + 1e-6))
    assert np.all(np.max(np.abs(vals), axis=1) == 448.0)


def test_e4m3_expert_is_the_plain_expert_on_e4m3_exact_operands():
    # X rows hold one entry 448 (scale 1); W1 makes a = 448 * 1 so that
    # silu(a) = a in fp64 (exp(-448) vanishes beside 1); W3 = c / 448^2 makes
    # h = c, e4m3 values with max |c| = 448 per row, so both quantizations are
    # exact and the FP8 expert equals the plain one bit for bit
    vals, _ = _e4m3_table()
    rng = np.random.default_rng(44)
    d, f, n = 8, 16, 8
    X = np.zeros((n, d))
    X[np.arange(n), np.arange(n) % d] = 448.0
    W1 = np.ones((d, f)) / 1.0
    c = rng.choice(vals[np.abs(vals) <= 448], size=(d, f))
    c[:, 0] = 448.0
    W3 = c / 448.0 ** 2
    W2 = rng.standard_normal((f, 4))
    plain = O.swiglu(X, W1, W3, W2, "f64")
    fp8 = O.swiglu(X, W1, W3, W2, "f64", act_e4m3=True)
    assert np.array_equal(plain, fp8)
    # on general operands the two differ, by the e4m3 rounding of the operands
    Xg = rng.standard_normal((n, d))
    a = O.swiglu(Xg, W1 * 0.3, W3 * 900, W2, "f64")
    b = O.swiglu(Xg, W1 * 0.3, W3 * 900, W2, "f64", act_e4m3=True)
    assert 0 < np.linalg.norm(a - b) / np.linalg.norm(a) < 0.1


def test_dequantize_e4m3_kmajor_is_the_transpose():
    rng = np.random.default_rng(45)
    qb = rng.integers(0, 126, size=(2, 5, 7)).astype(np.uint8)   # [S, K, n], finite codes
    sc = rng.uniform(0.5, 2, (2, 7))
    a = O.dequantize_e4m3(qb, sc)
    b = O.dequantize_e4m3(np.ascontiguousarray(np.swapaxes(qb, 1, 2)), sc, kmajor=True)
    assert np.array_equal(a, b)
    assert a[1, 3, 6] == O.e4m3_value(qb[1, 3, 6]) * sc[1, 6]


# ------------------------------------------------- device-level capacity (§2③)

def test_device_capacity_values():
    # finegrained layer: N_bar = 6*8192/64 = 768, a device of 8 experts holds 1.25*768*8
    assert O.device_capacity(1.25, 6, 8192, 64, 8, 6) == 7680
    assert O.device_capacity(math.inf, 6, 8192, 64, 8, 6) == 8192 * 6
    assert O.device_capacity(math.inf, 2, 100, 8, 1, 2) == 100
    for g in (0.5, 1.0, 1.5):  # one expert per device: the per-expert capacity
        assert O.device_capacity(g, 2, 4096, 8, 1, 2) == O.capacity(g, 2, 4096, 8)
    assert O.device_capacity(1e9, 2, 16, 8, 4, 3) == 16 * 3


def test_device_drop_with_one_expert_per_device_is_expert_drop():
    L = W.random_logits(300, 8, seed=31, quantum=0.25).numpy()
    L[:, 1] += 1.0
    for gamma in (0.5, 1.0, 1.3):
        a = O.route(L, mode="capacity_drop_device", k=2, N=8, gamma=gamma, group_size=1)
        b = O.route(L, mode="capacity_drop", k=2, N=8, gamma=gamma)
        for key in ("idx", "gate", "keep", "kept", "demand", "C"):
            assert np.array_equal(a[key], b[key]), key


def _brute_keep_device(cands, C):
    """cands: list of (token, slot, gate). The kept set is the unique C-subset
    whose members all rank above every non-member, rank = (gate desc, token
    asc, slot asc)."""
    if len(cands) <= C:
        return set((t, j) for t, j, _ in cands)
    def above(a, b):
        return (a[2] > b[2]) or (a[2] == b[2] and (a[0], a[1]) < (b[0], b[1]))
    best = None
    for sub in itertools.combinations(range(len(cands)), C):
        inside = [cands[i] for i in sub]
        outside = [cands[i] for i in range(len(cands)) if i not in sub]
        if all(above(a, b) for a in inside for b in outside):
            assert best is None
            best = set((t, j) for t, j, _ in inside)
    return best


@pytest.mark.parametrize("seed", range(4))
def test_device_drop_brute_force(seed):
    T, N, k, gs = 8, 4, 2, 2
    L = W.random_logits(T, N, seed=40 + seed, quantum=0.5).numpy()
    rt = O.route(L, mode="capacity_drop_device", k=k, N=N, gamma=0.75, group_size=gs)
    C = rt["C"]
    assert C == 6  # floor(0.75 * (2*8/4) * 2)
    for lo in range(0, N, gs):
        ts, js = np.nonzero((rt["idx"] >= lo) & (rt["idx"] < lo + gs))
        cands = [(int(t), int(j), float(rt["gate"][t, j])) for t, j in zip(ts, js)]
        kept = set((int(t), int(j)) for t, j in zip(ts, js) if rt["keep"][t, j])
        assert kept == _brute_keep_device(cands, C)
    for e in range(N):
        assert rt["kept"][e] == (rt["keep"] & (rt["idx"] == e)).sum()
        assert rt["demand"][e] == (rt["idx"] == e).sum()


def test_device_drop_invariants_and_room_sharing():
    T, N, k, gs = 2000, 16, 2, 4
    L = W.random_logits(T, N, seed=23, quantum=0.25).numpy()
    L[:, 0] += 2.0                                      # overload expert 0 of device 0
    dev = O.route(L, mode="capacity_drop_device", k=k, N=N, gamma=1.0, group_size=gs, renorm=True)
    per = O.route(L, mode="capacity_drop", k=k, N=N, gamma=1.0, renorm=True)
    Cd, Ce = dev["C"], per["C"]
    assert Cd == gs * Ce
    gk = O.key32(dev["gate"]).astype(np.int64)
    for lo in range(0, N, gs):
        ts, js = np.nonzero((dev["idx"] >= lo) & (dev["idx"] < lo + gs))
        kp = dev["keep"][ts, js]
        assert kp.sum() == min(len(ts), Cd)
        if (~kp).any() and kp.any():
            kk, dk = gk[ts[kp], js[kp]], gk[ts[~kp], js[~kp]]
            assert kk.min() >= dk.max()
            thr = kk.min()
            if (dk == thr).any():  # at the threshold key, kept (token, slot) precede dropped
                fk = (ts[kp] * k + js[kp])[kk == thr]
                fd = (ts[~kp] * k + js[~kp])[dk == thr]
                assert fk.max() < fd.min()
    # the device keeps at least as many pairs as its experts would alone, and
    # the overloaded expert uses room its device-mates leave
    assert dev["kept"].sum() >= per["kept"].sum()
    assert dev["kept"][0] > Ce and per["kept"][0] == Ce
    assert np.array_equal(dev["idx"], per["idx"]) and np.array_equal(dev["gate"], per["gate"])


def test_device_drop_unlimited_is_token_choice():
    L = W.random_logits(100, 8, seed=9).numpy()
    a = O.route(L, mode="capacity_drop_device", k=2, N=8, gamma=math.inf, group_size=4)
    b = O.route(L, mode="token_choice", k=2, N=8)
    for key in ("idx", "gate", "keep", "kept", "demand"):
        assert np.array_equal(a[key], b[key])

@pytest.mark.parametrize("quantum", [None, 0.25])
def test_expert_choice_invariants(quantum):
    T, N, k = 64, 8, 2
    L = W.random_logits(T, N, seed=8, quantum=quantum).numpy()
    rt = O.route(L, mode="expert_choice", k=k, N=N)
    c = k * T // N
    assert rt["C"] == c
    assert np.all(rt["keep"].sum(0) == c)
    assert rt["coverage"].sum() == N * c
    for e in range(N):
        col = rt["p"][:, e]
        sel = rt["keep"][:, e]
        brute = sorted(range(T), key=lambda t: (-float(col[t]), t))[:c]
        assert set(np.nonzero(sel)[0].tolist()) == set(brute)
        assert col[sel].min() >= col[~sel].max()


def test_expanded_candidates_local_and_disjoint():
    T, N, k, m, gs = 64, 16, 2, 3, 4
    L = W.random_logits(T, N, seed=9, quantum=0.5).numpy()
    base = O.topk_experts(L, k)
    ext = O.expanded_candidates(L, base, m, gs)
    hg = O.home_groups(T, N // gs)
    for t in range(T):
        g = int(hg[t])
        extra = [e for e in ext[t, k:].tolist() if e >= 0]
        members = set(range(g * gs, (g + 1) * gs))
        assert set(extra) <= members
        assert not set(extra) & set(base[t].tolist())
        pool = [e for e in sorted(members) if e not in set(base[t].tolist())]
        assert extra == _brute_topk_subset(L[t], pool, m)
    assert np.array_equal(O.expanded_candidates(L, base, 0, gs), base)


def _brute_topk_subset(row, pool, m):
    return sorted(pool, key=lambda e: (-float(row[e]), e))[:m]


def test_dispatch_bijection_and_order():
    T, N = 200, 8
    L = W.random_logits(T, N, seed=11).numpy()
    rt = O.route(L, mode="capacity_drop", k=2, N=N, gamma=1.0)
    dp = O.dispatch(rt["idx"], rt["gate"], rt["keep"], N)
    off, rtok = dp["expert_offsets"], dp["row_token"]
    assert off[0] == 0 and np.all(np.diff(off) == rt["kept"])
    seen = set()
    for e in range(N):
        toks = rtok[off[e]:off[e + 1]]
        assert np.all(np.diff(toks) > 0)
        for t in toks:
            j = np.nonzero(rt["idx"][t] == e)[0][0]
            assert rt["keep"][t, j]
            seen.add((int(t), e))
    assert len(seen) == int(rt["keep"].sum()) == dp["P"]
    for t in range(T):
        rows = [r for r in dp["tok_rows"][t].tolist() if r >= 0]
        assert rows == sorted(rows) and len(rows) == rt["keep"][t].sum()
        assert all(rtok[r] == t for r in rows)


# -------------------------------------------------------------- worked examples

def test_golden_routing_examples(golden_dir):
    with open(os.path.join(golden_dir, "routing_worked_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for case in cases:
        L = np.array(case["logits"], F32)
        rt = O.route(L, mode=case["mode"], k=case["k"], N=case["N"], gamma=_gamma(case["gamma"]),
                     m=case.get("m", 0), group_size=case.get("group_size", 8),
                     renorm=case["renorm"])
        exp = case["expected"]
        for key, val in exp.items():
            got = rt[key]
            if key == "C":
                assert got == val, case["name"]
            else:
                assert np.array_equal(np.asarray(got), np.asarray(val)), (case["name"], key, got)


def test_golden_swiglu_closed_form(golden_dir):
    with open(os.path.join(golden_dir, "swiglu_expert_closed_form.json")) as fh:
        c = json.load(fh)
    x = np.array(c["x"])
    out = O.layer_forward(x, np.zeros((2, 1)), None, np.array(c["W1"]), np.array(c["W3"]),
                          np.array(c["W2"]), mode="token_choice", k=1, dtype="f64")
    assert np.allclose(out["y"], np.array(c["expected_y"]), rtol=1e-15, atol=0)
    assert O.silu(np.array([0.0, 1.0, -1.0])).tolist() == pytest.approx(
        [0.0, 0.7310585786300049, -0.2689414213699951], rel=1e-15)


# ------------------------------------------------------------- experts, combine

def _tiny_layer(seed, d=12, f=20, N=4, T=24, dtype="f64"):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g, dtype=torch.float64).numpy()
    Wr = torch.randn(d, N, generator=g, dtype=torch.float64).numpy() / math.sqrt(d)
    W1 = torch.randn(N, d, f, generator=g, dtype=torch.float64).numpy() / math.sqrt(d)
    W3 = torch.randn(N, d, f, generator=g, dtype=torch.float64).numpy() / math.sqrt(d)
    W2 = torch.randn(N, f, d, generator=g, dtype=torch.float64).numpy() / math.sqrt(f)
    return x, Wr, W1, W3, W2


@pytest.mark.parametrize("mode,gamma", [("token_choice", math.inf), ("capacity_drop", 1.0),
                                        ("expert_choice", math.inf)])
def test_sparse_layer_equals_dense_then_mask(mode, gamma):
    """Apply every expert to every token densely, weight by G masked to the
    kept pairs, and sum: the layer equation read literally."""
    x, Wr, W1, W3, W2 = _tiny_layer(12)
    T, N = x.shape[0], W1.shape[0]
    out = O.layer_forward(x, Wr, None, W1, W3, W2, mode=mode, k=2, gamma=gamma, dtype="f64",
                          renorm=(mode == "token_choice"))
    G = np.zeros((T, N))
    for t in range(T):
        for j in range(out["idx"].shape[1]):
            if out["keep"][t, j]:
                G[t, out["idx"][t, j]] = out["gate"][t, j]
    dense = np.stack([(torch.nn.functional.silu(torch.from_numpy(x @ W1[e])) *
                       torch.from_numpy(x @ W3[e])).numpy() @ W2[e] for e in range(N)], 1)
    y = np.einsum("te,ted->td", G, dense)
    assert np.allclose(out["y"], y, rtol=1e-12, atol=1e-12)


def test_expert_choice_c_equals_T_is_dense_softmax_mixture():
    x, Wr, W1, W3, W2 = _tiny_layer(13, N=4, T=8)
    # k = N makes c = k*T/N = T: every expert takes every token
    out = O.layer_forward(x, Wr, None, W1, W3, W2, mode="expert_choice", k=4, dtype="f64")
    assert out["keep"].all()
    L = x @ Wr
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    dense = np.stack([(torch.nn.functional.silu(torch.from_numpy(x @ W1[e])) *
                       torch.from_numpy(x @ W3[e])).numpy() @ W2[e] for e in range(4)], 1)
    y = np.einsum("te,ted->td", p, dense)
    assert np.allclose(out["y"], y, rtol=1e-6, atol=1e-7)


def test_single_expert_is_dense_swiglu_ffn():
    x, Wr, W1, W3, W2 = _tiny_layer(14, N=1)
    out = O.layer_forward(x, Wr[:, :1], None, W1, W3, W2, mode="token_choice", k=1, dtype="f64")
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0])) *
           (xt @ torch.from_numpy(W3[0]))) @ torch.from_numpy(W2[0])
    assert np.allclose(out["y"], ref.numpy(), rtol=1e-13, atol=1e-13)


def test_shared_expert_added_with_gate_one_and_zero_coverage_tokens():
    x, Wr, W1, W3, W2 = _tiny_layer(15, N=4, T=16)
    g = torch.Generator().manual_seed(99)
    d, fs = x.shape[1], 10
    Ws1 = torch.randn(d, fs, generator=g, dtype=torch.float64).numpy()
    Ws3 = torch.randn(d, fs, generator=g, dtype=torch.float64).numpy()
    Ws2 = torch.randn(fs, d, generator=g, dtype=torch.float64).numpy()
    base = O.layer_forward(x, Wr, None, W1, W3, W2, mode="capacity_drop", k=2, gamma=0.0,
                           dtype="f64")
    assert np.all(base["y"] == 0.0)                 # every pair dropped: y = 0
    sh = O.layer_forward(x, Wr, None, W1, W3, W2, mode="capacity_drop", k=2, gamma=0.0,
                         dtype="f64", Ws1=Ws1, Ws3=Ws3, Ws2=Ws2)
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(Ws1)) *
           (xt @ torch.from_numpy(Ws3))) @ torch.from_numpy(Ws2)
    assert np.allclose(sh["y"], ref.numpy(), rtol=1e-13, atol=1e-13)


def test_token_subset_matches_full_batch():
    x, Wr, W1, W3, W2 = _tiny_layer(16, N=4, T=30)
    full = O.layer_forward(x, Wr, None, W1, W3, W2, mode="capacity_drop", k=2, gamma=1.0,
                           dtype="bf16")
    sub = O.layer_forward(x, Wr, None, W1, W3, W2, mode="capacity_drop", k=2, gamma=1.0,
                          dtype="bf16", tokens=[3, 17, 29])
    assert np.array_equal(sub["y"], full["y"][[3, 17, 29]])


# ------------------------------------------------------------------ statistics

def test_balance_statistic_closed_forms():
    L = W.random_logits(64, 8, seed=17).numpy()
    ec = O.route(L, mode="expert_choice", k=2, N=8)
    s = O.load_stats(ec["demand"], ec["kept"], ec["p"])
    # expert choice: f_i = 1/N, so B = (1/N) sum_i P_i = 1/N
    assert s["balance_times_N"] == pytest.approx(1.0, abs=1e-6)
    assert s["max_over_mean"] == 1.0 and s["drop_fraction"] == 0.0
    uni = O.route(np.zeros((16, 4), F32), mode="token_choice", k=1, N=4)
    s = O.load_stats(uni["demand"], uni["kept"], uni["p"])
    # all ties: every token picks expert 0; f = (1,0,0,0), P = 1/4 each
    assert uni["demand"].tolist() == [16, 0, 0, 0]
    assert s["balance"] == pytest.approx(0.25) and s["max_over_mean"] == 4.0


def test_workload_recipe_shapes_and_zipf():
    w = W.TINY_F32
    inp = W.make_inputs(w)
    assert inp["x"].shape == (256, 128) and inp["W1"].shape == (8, 128, 256)
    assert inp["W2"].shape == (8, 256, 128) and inp["x"].dtype == torch.float32
    b = W.zipf_log_probs(8, 1.2).astype(np.float64)
    p = np.exp(b)
    assert abs(p.sum() - 1) < 1e-6 and np.all(np.diff(b) < 0)
    assert p[0] / p[1] == pytest.approx(2 ** 1.2, rel=1e-5)
    again = W.make_inputs(w)
    assert torch.equal(inp["x"], again["x"]) and torch.equal(inp["W2"], again["W2"])
