"""moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate
device memory (a framework that hands an operator only its inputs and
outputs, or a loop where cudaMalloc may not run). It keeps the SwiGLU hidden
activations in the library's own static device array instead of a caller
workspace. Checked through the C ABI against moe_expert_ffn on two calls in a
row with different data, so the second call cannot pass on the first call's
leftovers. Collected last on purpose: it also runs alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import routing_capacity_drop_router_b300 as M
from tests import gpu_util as G


def _case(seed, sizes, d, f, dtype):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    S = len(sizes)
    off = np.zeros(S + 1, dtype=np.int32)
    off[1:] = np.cumsum(sizes)
    rows_max = int(off[-1]) + 3
    xp = torch.randn((rows_max, d), generator=g).to(dt)
    W1 = (torch.randn((S, d, f), generator=g) * d ** -0.5).to(dt)
    W3 = (torch.randn((S, d, f), generator=g) * d ** -0.5).to(dt)
    W2 = (torch.randn((S, f, d), generator=g) * f ** -0.5).to(dt)
    dev = torch.device("cuda")
    return dict(off=torch.from_numpy(off).to(dev), S=S, rows_max=rows_max, P=int(off[-1]),
                xp=xp.to(dev), W1=W1.to(dev), W3=W3.to(dev), W2=W2.to(dev), dt=dt)


def _with_workspace(cfg, c, f):
    op = torch.zeros((c["rows_max"], cfg.d), dtype=c["dt"], device="cuda")
    ws = torch.zeros(M.ffn_workspace_size(c["rows_max"], f, cfg.dtype), dtype=torch.uint8,
                     device="cuda")
    M.moe_expert_ffn(cfg, c["xp"], c["off"], c["S"], c["rows_max"], f, c["W1"], c["W3"], c["W2"],
                     op, ws)
    return op


def _without_workspace(cfg, c, f, status):
    op = torch.zeros((c["rows_max"], cfg.d), dtype=c["dt"], device="cuda")
    M.moe_expert_ffn_noalloc(cfg, c["xp"], c["off"], c["S"], c["rows_max"], f, c["W1"], c["W3"],
                             c["W2"], op, device_status=status)
    return op


@pytest.fixture(params=["one_cta", "cta_pairs"])
def gemm_form(request, monkeypatch):
    """Both forms of the bf16 grouped GEMM run through the static array."""
    monkeypatch.setenv("MOE_GEMM_CTA_PAIRS", "1" if request.param == "cta_pairs" else "0")
    return request.param


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,d,f,calls", [
    ("bf16", 256, 384, ((1, [130, 0, 257, 9]), (2, [1, 300, 64, 200]))),
    # segments of several 256-row pair tiles, each with a ragged tail
    ("bf16", 256, 384, ((4, [700, 0, 913, 433]), (5, [1030, 257, 1, 640]))),
    ("f32", 128, 192, ((1, [130, 0, 257, 9]), (2, [1, 300, 64, 200]))),
])
def test_noalloc_matches_workspace_entry_point_twice(dtype, d, f, calls, gemm_form):
    """The same kernels run on the same data, so the two entry points agree
    bit for bit; two calls in a row with different data, so the second call
    cannot pass on the first call's leftovers in the shared array."""
    cfg = M.make_config(T=1, d=d, N=4, f=f, k=1, dtype=dtype)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for seed, sizes in calls:
        c = _case(seed, sizes, d, f, dtype)
        ref = _with_workspace(cfg, c, f)
        got = _without_workspace(cfg, c, f, status)
        torch.cuda.synchronize()
        assert int(status.item()) == M.MOE_OK
        P = c["P"]
        assert torch.equal(got[:P], ref[:P]), f"call with seed {seed} differs"
        G.assert_output_close(G.np32(got[:P]), G.np32(ref[:P]).astype(np.float64), dtype,
                              f"call with seed {seed}")
        assert torch.all(got[P:] == 0)


@pytest.mark.gpu
def test_noalloc_leaves_the_callers_status_word_alone():
    """A word that already holds an earlier stage's error keeps it."""
    cfg = M.make_config(T=1, d=128, N=2, f=128, k=1, dtype="bf16")
    c = _case(6, [100, 50], 128, 128, "bf16")
    status = torch.full((1,), M.MOE_ERR_DEVICE_BOUNDS, dtype=torch.int32, device="cuda")
    ref = _with_workspace(cfg, c, 128)
    got = _without_workspace(cfg, c, 128, status)
    torch.cuda.synchronize()
    assert int(status.item()) == M.MOE_ERR_DEVICE_BOUNDS
    assert torch.equal(got[:c["P"]], ref[:c["P"]])


@pytest.mark.gpu
def test_noalloc_without_status_pointer():
    cfg = M.make_config(T=1, d=128, N=2, f=128, k=1, dtype="bf16")
    c = _case(3, [100, 50], 128, 128, "bf16")
    ref = _with_workspace(cfg, c, 128)
    got = _without_workspace(cfg, c, 128, None)
    torch.cuda.synchronize()
    assert torch.equal(got[:c["P"]], ref[:c["P"]])


def test_noalloc_rejects_sizes_beyond_its_array():
    # checked on the host before any CUDA call, so no GPU is needed
    cfg = M.make_config(T=1, d=4096, N=8, f=14336, k=1, dtype="bf16")
    fake = 0x10000
    limit_rows = (M.MOE_NOALLOC_SCRATCH_BYTES - 256) // (14336 * 2)
    st = M.lib().moe_expert_ffn_noalloc(ctypes.byref(cfg), fake, fake, 8, limit_rows + 1, 14336,
                                        fake, fake, fake, fake, None, None)
    assert st == M.MOE_ERR_WORKSPACE
