"""The C ABI library: loads, exports every entry point of include/moe.h, sizes
its buffers as the capacity formulas say, and rejects bad arguments on the
host before any CUDA call (so these run without a GPU)."""
import ctypes
import math
import os
import re

import pytest

import moe_workloads as W
import oracle as O
import routing_capacity_drop_router_b300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|void|const char\*)\s+(moe_\w+)\s*\(", src,
                                 flags=re.M)))


def test_library_exports_every_declared_entry_point():
    names = _declared_functions()
    assert len(names) >= 16
    lib = M.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(M.SIGNATURES), "binding and header disagree"


def test_struct_layout_matches_header():
    assert ctypes.sizeof(M.moe_config) == 56
    assert M.moe_config.gamma.offset == 24
    assert ctypes.sizeof(M.moe_sizes_t) == 32
    assert ctypes.sizeof(M.moe_views_t) == 17 * 8
    assert ctypes.sizeof(M.moe_e4m3_experts) == 6 * 8


@pytest.mark.parametrize("w", list(W.ALL.values()), ids=list(W.ALL))
def test_sizes_follow_capacity_formulas(w):
    s = M.sizes(M.config_from_workload(w))
    if w.mode == W.EXPERT_CHOICE:
        c = O.ec_capacity(w.k, w.T, w.N)
        assert (s.kc, s.capacity, s.rows_max) == (w.N, c, w.N * c)
    elif w.mode == W.CAPACITY_DROP:
        C = O.capacity(w.gamma, w.k, w.T, w.N)
        assert (s.kc, s.capacity) == (w.k + w.m, C)
        assert s.rows_max == min(w.T * (w.k + w.m), w.N * C)
    elif w.mode == W.CAPACITY_DROP_DEVICE:
        kc = w.k + w.m
        C = O.device_capacity(w.gamma, w.k, w.T, w.N, w.group_size, kc)
        assert (s.kc, s.capacity) == (kc, C)
        assert s.rows_max == min(w.T * kc, (w.N // w.group_size) * C)
    else:
        assert (s.kc, s.capacity, s.rows_max) == (w.k + w.m, w.T, w.T * (w.k + w.m))
    assert s.workspace > 0 and M.workspace_size(M.config_from_workload(w)) == s.workspace


@pytest.mark.parametrize("gamma", [0.0, 0.7, 1.0, 1.25, 3.0, math.inf])
@pytest.mark.parametrize("gs", [1, 2, 4, 8])
def test_device_capacity_matches_oracle(gamma, gs):
    w = W.Workload("dev", T=1000, d=64, N=8, f=64, k=3, mode=W.CAPACITY_DROP_DEVICE,
                   gamma=gamma, group_size=gs, m=1)
    s = M.sizes(M.config_from_workload(w))
    assert s.capacity == O.device_capacity(gamma, 3, 1000, 8, gs, 4)


def test_device_drop_needs_a_group_that_divides_N():
    for gs in (0, 3, 16):
        cfg = M.make_config(T=64, d=64, N=8, f=64, k=2, mode="capacity_drop_device", gamma=1.0,
                            group_size=gs)
        with pytest.raises(M.MoeError) as ei:
            M.sizes(cfg)
        assert ei.value.status == M.MOE_ERR_SHAPE


def test_workload_capacities_match_the_pages_formulas():
    assert M.sizes(M.config_from_workload(W.mixtral(1.0))).capacity == 1024
    assert M.sizes(M.config_from_workload(W.mixtral(1.5))).capacity == 1536
    assert M.sizes(M.config_from_workload(W.FINE_BF16)).capacity == 960
    assert M.sizes(M.config_from_workload(W.EC_BF16)).capacity == 256


def _cfg(**kw):
    base = dict(T=64, d=128, N=8, f=128, k=2)
    base.update(kw)
    return M.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), M.MOE_ERR_SHAPE),
    (dict(k=9), M.MOE_ERR_SHAPE),
    (dict(d=100), M.MOE_ERR_SHAPE),               # bf16 needs d % 64 == 0
    (dict(f=96), M.MOE_ERR_SHAPE),
    (dict(N=300, k=2), M.MOE_ERR_UNSUPPORTED),
    (dict(T=100000), M.MOE_ERR_UNSUPPORTED),
    (dict(N=64, k=20, m=20, group_size=8), M.MOE_ERR_UNSUPPORTED),
    (dict(gamma=float("nan"), mode="capacity_drop"), M.MOE_ERR_SHAPE),
    (dict(gamma=-1.0, mode="capacity_drop"), M.MOE_ERR_SHAPE),
    (dict(m=2, group_size=3), M.MOE_ERR_SHAPE),
    (dict(mode=7), M.MOE_ERR_SHAPE),
    (dict(dtype=5), M.MOE_ERR_SHAPE),
])
def test_invalid_configs_are_rejected(kw, code):
    cfg = _cfg(**kw)
    out = M.moe_sizes_t()
    assert M.lib().moe_sizes(ctypes.byref(cfg), ctypes.byref(out)) == code
    assert M.lib().moe_workspace_size(ctypes.byref(cfg)) == 0


def test_null_pointers_rejected_before_any_launch():
    lib = M.lib()
    cfg = _cfg()
    r = ctypes.byref(cfg)
    assert lib.moe_route(r, *([None] * 9), 0, None) == M.MOE_ERR_NULL
    assert lib.moe_capacity_drop(r, None, None, None, None, None, None, None) == M.MOE_ERR_NULL
    assert lib.moe_dispatch(r, *([None] * 11), None) == M.MOE_ERR_NULL
    assert lib.moe_combine(r, None, None, None, None, None, None) == M.MOE_ERR_NULL
    assert lib.moe_layer_forward(r, *([None] * 14), 0, None) == M.MOE_ERR_NULL
    assert lib.moe_expert_ffn(r, None, None, 8, 64, 128, None, None, None, None, None, 0,
                              None) == M.MOE_ERR_NULL
    assert lib.moe_load_stats(r, None, None, None, None, None, 0, None) == M.MOE_ERR_NULL
    assert lib.moe_get_device_status(None, None, None) == M.MOE_ERR_NULL
    assert lib.moe_route(None, *([None] * 9), 0, None) == M.MOE_ERR_NULL
    assert lib.moe_route_workspace_size(None) == 0


def test_misaligned_and_small_workspace_rejected_before_any_launch():
    lib = M.lib()
    cfg = _cfg()
    r = ctypes.byref(cfg)
    fake = 0x10000  # never dereferenced: the checks fail first
    ptrs = [fake] * 6
    # x misaligned
    assert lib.moe_layer_forward(r, fake + 2, fake, None, fake, fake, fake, None, None, None, None,
                                 None, fake, None, fake, 1 << 40, None) == M.MOE_ERR_ALIGN
    # workspace below moe_workspace_size
    need = lib.moe_workspace_size(r)
    assert lib.moe_layer_forward(r, fake, fake, None, fake, fake, fake, None, None, None, None,
                                 None, fake, None, fake, need - 1, None) == M.MOE_ERR_WORKSPACE
    # given logits flag without logits
    cfg2 = _cfg(logits_given=True)
    assert lib.moe_layer_forward(ctypes.byref(cfg2), fake, None, None, fake, fake, fake, None, None,
                                 None, None, None, fake, None, fake, need, None) == M.MOE_ERR_NULL
    assert lib.moe_expert_ffn(r, fake, fake, 8, 64, 128, *ptrs[:4], fake, 10, None) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_grouped_gemm(M.MOE_BF16, fake, fake, 8, 64, 100, 128, fake, fake, fake, 1 << 20,
                                None) == M.MOE_ERR_SHAPE
    # moe_load_stats: 8 * N * ceil(T / 32) scratch bytes; a misaligned scratch of
    # exactly that size passes the size check and fails the alignment one
    stats_need = 8 * cfg.N * -(-cfg.T // 32)
    assert lib.moe_load_stats(r, fake, fake, fake, fake, fake, stats_need - 1, None) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_load_stats(r, fake, fake, fake, fake, fake + 8, stats_need, None) == \
        M.MOE_ERR_ALIGN


def test_expert_ffn_on_sms_host_checks():
    lib = M.lib()
    fake = ctypes.c_void_p(1 << 20)
    bf = M.make_config(T=8, d=64, N=2, f=64, k=1, dtype="bf16")
    f32 = M.make_config(T=8, d=64, N=2, f=64, k=1, dtype="f32")
    args = [fake, fake, 2, 8, 64, fake, fake, fake, fake]
    need = M.ffn_workspace_size(8, 64, "bf16")
    assert lib.moe_expert_ffn_on_sms(ctypes.byref(f32), *args, 4, fake, need, None) == \
        M.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_on_sms(ctypes.byref(bf), *args, 0, fake, need, None) == \
        M.MOE_ERR_SHAPE
    assert lib.moe_expert_ffn_on_sms(ctypes.byref(bf), *args, 4, None, need, None) == \
        M.MOE_ERR_NULL
    assert lib.moe_expert_ffn_on_sms(ctypes.byref(bf), *args, 4, fake, need - 1, None) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_expert_ffn_on_sms(None, *args, 4, fake, need, None) == M.MOE_ERR_NULL


def test_expert_ffn_gather_host_checks():
    """moe_expert_ffn_gather rejects every bad argument before any launch."""
    lib = M.lib()
    fake = ctypes.c_void_p(1 << 20)
    bf = M.make_config(T=8, d=64, N=2, f=64, k=1, dtype="bf16")
    f32 = M.make_config(T=8, d=64, N=2, f=64, k=1, dtype="f32")
    odd = M.make_config(T=8, d=96, N=2, f=64, k=1, dtype="bf16")
    need = M.ffn_workspace_size(8, 64, "bf16")

    def call(cfg, x=fake, row_token=fake, ws=fake, ws_bytes=need, f=64, W2=fake):
        return lib.moe_expert_ffn_gather(cfg, x, row_token, fake, 2, 8, f, fake, fake, W2, fake,
                                         ws, ws_bytes, None)

    assert call(ctypes.byref(f32)) == M.MOE_ERR_UNSUPPORTED
    assert call(ctypes.byref(odd)) == M.MOE_ERR_SHAPE
    assert call(ctypes.byref(bf), f=100) == M.MOE_ERR_SHAPE
    assert call(None) == M.MOE_ERR_NULL
    assert call(ctypes.byref(bf), x=None) == M.MOE_ERR_NULL
    assert call(ctypes.byref(bf), row_token=None) == M.MOE_ERR_NULL
    assert call(ctypes.byref(bf), W2=None) == M.MOE_ERR_NULL
    assert call(ctypes.byref(bf), x=ctypes.c_void_p((1 << 20) + 8)) == M.MOE_ERR_ALIGN
    assert call(ctypes.byref(bf), ws_bytes=need - 1) == M.MOE_ERR_WORKSPACE


def test_fuse_gather_flag_in_config():
    cfg = M.make_config(T=8, d=64, N=2, f=64, k=1, fuse_gather=True, logits_given=True)
    assert cfg.flags == M.MOE_FUSE_GATHER | M.MOE_LOGITS_GIVEN
    assert M.sizes(cfg).workspace == M.sizes(M.make_config(T=8, d=64, N=2, f=64, k=1)).workspace


def test_e4m3_experts_host_checks():
    lib = M.lib()
    fake = ctypes.c_void_p(1 << 20)
    ex = M.moe_e4m3_experts(*([1 << 20] * 6))
    need = M.ffn_workspace_size_e4m3(8, 128, 128)
    args = lambda cfg, f, e: (ctypes.byref(cfg), fake, fake, 2, 8, f, e, fake, fake, need, None)  # noqa: E731
    bf = M.make_config(T=8, d=128, N=2, f=128, k=1, dtype="bf16")
    f32 = M.make_config(T=8, d=128, N=2, f=128, k=1, dtype="f32")
    assert lib.moe_expert_ffn_e4m3(*args(f32, 128, ctypes.byref(ex))) == M.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_e4m3(*args(bf, 192, ctypes.byref(ex))) == M.MOE_ERR_SHAPE
    assert lib.moe_expert_ffn_e4m3(*args(bf, 128, None)) == M.MOE_ERR_NULL
    bad = M.moe_e4m3_experts(*([1 << 20] * 5 + [None]))
    assert lib.moe_expert_ffn_e4m3(*args(bf, 128, ctypes.byref(bad))) == M.MOE_ERR_NULL
    assert lib.moe_layer_forward_e4m3(ctypes.byref(bf), *([None] * 3), None, *([None] * 8), 0,
                                      None) == M.MOE_ERR_NULL


def test_e4m3_workspace_sizes():
    # control block, bf16 hidden rows, e4m3 token rows + scales, e4m3 hidden rows + scales
    a = lambda n: (n + 255) // 256 * 256  # noqa: E731
    R, d, f = 1000, 4096, 14336
    assert M.ffn_workspace_size_e4m3(R, d, f) == \
        M.MOE_CTRL_BYTES + a(R * f * 2) + a(R * d) + a(R * 4) + a(R * f) + a(R * 4)
    cfg = M.make_config(T=64, d=256, N=8, f=512, k=2)
    R = M.sizes(cfg).rows_max
    assert M.workspace_size_e4m3(cfg) == M.workspace_size(cfg) + a(R * 256) + a(R * 4) + \
        a(R * 512) + a(R * 4)
    assert M.workspace_size_e4m3(M.make_config(T=64, d=256, N=300, f=512, k=2)) == 0


def test_status_strings():
    for code in range(-8, 1):
        assert M.status_string(code) and M.status_string(code) != "unknown status"
    assert M.status_string(-99) == "unknown status"


def test_layer_stage_list_follows_the_config():
    names = M.moe_layer_stages(_cfg())
    assert names == ["router", "select", "dispatch", "expert_gemm1_swiglu", "expert_gemm2",
                     "combine"]
    names = M.moe_layer_stages(_cfg(f_shared=128, logits_given=True))
    assert names == ["route_tokens", "select", "dispatch", "expert_gemm1_swiglu", "expert_gemm2",
                     "shared_offsets", "shared_gemm1_swiglu", "shared_gemm2", "combine"]
    names = M.moe_layer_stages(_cfg(dtype="f32"))
    assert names[:2] == ["router_logits", "route_tokens"]
    assert M.lib().moe_layer_stages(ctypes.byref(_cfg(N=0)), None, 0) == M.MOE_ERR_SHAPE
    # the fused gather launches the same six kernels (dispatch keeps the row tables)
    assert M.moe_layer_stages(_cfg(fuse_gather=True)) == M.moe_layer_stages(_cfg())


def test_trace_event_arguments_checked_on_the_host():
    lib = M.lib()
    assert lib.moe_set_trace_events(None, 0) == M.MOE_OK
    assert lib.moe_set_trace_events(None, 3) == M.MOE_ERR_NULL
    assert lib.moe_set_trace_events(None, -1) == M.MOE_ERR_SHAPE
    handles = (ctypes.c_void_p * 40)()
    assert lib.moe_set_trace_events(handles, 33) == M.MOE_ERR_SHAPE
    assert lib.moe_set_trace_events(handles, 2) == M.MOE_OK  # NULL entries: no event there
    assert lib.moe_set_trace_events(None, 0) == M.MOE_OK
