"""Host-side arithmetic of bench.py: the algorithmic bytes and flops the
roofline divides by (per-unit formulas of the kernel table), and the oracle
sampler's bounded sample. No GPU."""
import numpy as np
import pytest

import bench
import moe_workloads as W


def test_stage_bytes_follow_the_per_unit_formulas():
    w = W.ALL["mixtral_bf16_gamma1"]
    P = 4916
    b = bench.stage_bytes(w, P)
    s = 2
    assert b["route"] == w.T * w.d * s + w.d * w.N * s + w.T * w.N * 8 + w.T * (w.k + w.m) * 8
    assert b["dispatch"] == w.T * w.d * s + P * w.d * s + 16 * P
    assert b["combine"] == P * w.d * s + w.T * w.d * s + 8 * P
    # the gather fused into GEMM1: dispatch writes only the row tables
    f = bench.stage_bytes(w, P, fused_gather=True)
    assert f["dispatch"] == 16 * P
    assert f["route"] == b["route"] and f["combine"] == b["combine"]
    # a shared expert's output is read once more by the combine
    g = W.ALL["finegrained_bf16"]
    assert bench.stage_bytes(g, 100)["combine"] == 100 * g.d * 2 + 2 * g.T * g.d * 2 + 800


def test_routed_weight_bytes_count_the_experts_hit():
    w = W.ALL["decode_bf16"]
    kept = np.array([3, 0, 9, 1, 0, 0, 7, 2])
    assert bench.routed_weight_bytes(w, kept) == 5 * 3 * w.d * w.f * 2
    q = W.ALL["decode_e4m3"]
    per = 3 * q.d * q.f + 4 * (2 * q.f + q.d)  # e4m3 bytes + fp32 column scales
    assert bench.routed_weight_bytes(q, kept) == 5 * per


def test_ffn_flops_count_kept_pairs_and_the_shared_expert():
    w = W.ALL["mixtral_bf16_gamma1"]
    assert bench.ffn_flops(w, 10) == 6.0 * w.d * w.f * 10
    g = W.ALL["finegrained_bf16"]
    assert bench.ffn_flops(g, 10) == 6.0 * g.d * g.f * 10 + 6.0 * g.d * g.f_shared * g.T


@pytest.mark.parametrize("target_s", [0.05, 0.5])
def test_oracle_sampler_takes_a_bounded_sample(target_s):
    w = W.TINY_F32
    smp = bench.OracleSampler(w)
    n = smp.calibrate(target_s)
    assert 1 <= n <= w.T
    got, dt = smp.run(n)
    assert got == n and dt > 0
    assert "full-batch routing" in smp.describe(got, dt)


def test_vs_cublas_shapes_meet_the_grouped_gemm_shape_rules():
    """--vs-cublas runs moe_grouped_gemm, which takes bf16 K and n_out in
    multiples of 64 and at most 256 segments, and cuBLAS's batched form,
    which needs equal segments: every shape must satisfy both, and the
    first two must be the expert GEMMs of the Mixtral-shaped workload."""
    w = W.ALL["mixtral_bf16"]
    for S, n, K, n_out in bench.VS_CUBLAS_SHAPES:
        assert 1 <= S <= 256 and n >= 1
        assert K % 64 == 0 and n_out % 64 == 0
    (S1, n1, K1, o1), (S2, n2, K2, o2) = bench.VS_CUBLAS_SHAPES[:2]
    assert (S1, K1, o1) == (w.N, w.d, 2 * w.f) and (S2, K2, o2) == (w.N, w.f, w.d)
    assert n1 == n2 == w.k * w.T // w.N  # rows per expert with no capacity limit, on average
