"""GPU grouped expert GEMMs: the tcgen05 bf16 kernels against torch matmul and
the oracle's SwiGLU expert, the fp32 FMA kernels against the oracle at 1e-5,
over ragged segments (empty, one-row, several 128-row tiles, partial n-tiles)."""
import numpy as np
import pytest
import torch

import moe_workloads as W
import oracle as O
from tests import gpu_util as G

M = G.M
pytestmark = pytest.mark.gpu


def _segments(sizes):
    off = np.zeros(len(sizes) + 1, dtype=np.int32)
    off[1:] = np.cumsum(sizes)
    return off


@pytest.fixture(params=["cta_pairs", "cta_pairs_padded", "single_cta"])
def gemm_form(request, monkeypatch):
    """Run a bf16 case through every form of the tcgen05 grouped GEMM: CTA
    pairs (cta_group::2, 256-row tiles) whose segment tails run transposed,
    and every tile of the second GEMM (the default), the same pairs with no
    tile transposed and the tails padded to 256 rows, and one CTA per
    128-row tile."""
    monkeypatch.setenv("MOE_GEMM_CTA_PAIRS", "0" if request.param == "single_cta" else "1")
    monkeypatch.setenv("MOE_GEMM_SWAP_TAILS", "0" if request.param == "cta_pairs_padded" else "1")
    return request.param


# one segment per tail class of a 256-row pair tile: tails of 1..255 rows
# (a transposed tile's N = 32..256 after rounding up to 32; tails that end in
# either half of the pair's N/2 : N/2 token split), whole tiles, and a tile
# plus a tail
TAIL_SIZES = [1, 7, 8, 9, 15, 16, 17, 31, 33, 100, 127, 128, 129, 200, 240, 255, 256, 257, 513]


@pytest.mark.parametrize("K,n_out", [(192, 320), (1024, 256), (64, 64), (64, 448)])
def test_grouped_gemm_every_tail_class(K, n_out, gemm_form):
    """The grouped GEMM over segments of every tail size against fp64
    products; n_out = 320 leaves the last n-tile of each segment a quarter
    full, n_out = 64 is a single weight box (the second CTA of a pair holds no
    output column), K = 64 a single k-block. Rows past the last segment stay
    untouched."""
    _grouped_gemm_case(TAIL_SIZES, K, n_out)


@pytest.mark.parametrize("d,f", [(320, 192), (256, 1408)])
def test_expert_ffn_every_tail_class(d, f, gemm_form):
    """The SwiGLU expert over segments of every tail size against the oracle;
    f = 192 leaves GEMM1's last n-tile half full (a transposed tile's second
    CTA then holds no output column)."""
    _expert_ffn_case(TAIL_SIZES, d, f)


def _rand(shape, seed, scale=1.0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype)


@pytest.mark.parametrize("sizes,K,n_out", [
    ([130, 0, 170, 1, 249], 256, 320),
    ([128], 128, 256),
    ([3, 500, 64, 0, 0, 257], 512, 512),
    ([1000], 1024, 192),
    ([19150, 50], 512, 256),      # 151 tiles: one more than a full round of CTAs
    ([77, 300, 5], 2048, 512),    # few tiles, long K, ragged rows
])
def test_grouped_gemm_bf16_against_torch(sizes, K, n_out, gemm_form):
    _grouped_gemm_case(sizes, K, n_out)


def _grouped_gemm_case(sizes, K, n_out):
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P + 37
    A = _rand((rows_max, K), 1)
    B = _rand((S, K, n_out), 2, K ** -0.5)
    dev = torch.device("cuda")
    out = torch.full((rows_max, n_out), 7.0, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(M.ffn_workspace_size(0, 0, "bf16"), dtype=torch.uint8, device=dev)
    M.moe_grouped_gemm("bf16", A.cuda(), torch.from_numpy(off).cuda(), S, rows_max, K, n_out,
                       B.cuda(), out, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    got = out.float().cpu()
    for s in range(S):
        a, b = int(off[s]), int(off[s + 1])
        if a == b:
            continue
        ref = A[a:b].double() @ B[s].double()
        G.assert_output_close(got[a:b].numpy(), ref.numpy(), "bf16", f"segment {s}")
    assert torch.all(got[P:] == 7.0), "rows past the last segment were written"


@pytest.mark.parametrize("sizes,d,f", [
    ([130, 0, 170, 1, 249], 256, 384),
    ([300, 300], 320, 128),
    ([77], 2048, 1408),
])
def test_expert_ffn_bf16_against_oracle(sizes, d, f, gemm_form):
    _expert_ffn_case(sizes, d, f)


def _expert_ffn_case(sizes, d, f):
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P + 5
    xp = _rand((rows_max, d), 3)
    W1 = _rand((S, d, f), 4, d ** -0.5)
    W3 = _rand((S, d, f), 5, d ** -0.5)
    W2 = _rand((S, f, d), 6, f ** -0.5)
    cfg = M.make_config(T=1, d=d, N=S, f=f, k=1, dtype="bf16")
    dev = torch.device("cuda")
    op = torch.zeros((rows_max, d), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(M.ffn_workspace_size(rows_max, f, "bf16"), dtype=torch.uint8, device=dev)
    M.moe_expert_ffn(cfg, xp.cuda(), torch.from_numpy(off).cuda(), S, rows_max, f, W1.cuda(),
                     W3.cuda(), W2.cuda(), op, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    got = op.float().cpu().numpy()
    for s in range(S):
        a, b = int(off[s]), int(off[s + 1])
        if a == b:
            continue
        ref = O.swiglu(G.np32(xp[a:b]), G.np32(W1[s]), G.np32(W3[s]), G.np32(W2[s]), "bf16")
        G.assert_output_close(got[a:b], ref, "bf16", f"segment {s}")


@pytest.mark.parametrize("sizes,d,f,T", [
    ([130, 0, 170, 1, 249], 256, 384, 300),
    ([3, 500, 64, 0, 0, 257], 512, 256, 700),   # several 256-row tiles, empty segments
    ([77, 300, 5], 2048, 512, 200),             # long K: the row ring wraps many times
    ([1000], 128, 128, 1000),                   # one k-block per tile
])
def test_expert_ffn_gather_equals_copy(sizes, d, f, T, gemm_form):
    """moe_expert_ffn_gather on (x, row_token) computes the same bits as
    moe_expert_ffn on the copied rows xp[r] = x[row_token[r]] (tokens repeat,
    as under top-k), and matches the oracle; rows past the segments stay
    untouched."""
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P + 37
    x = _rand((T, d), 21)
    row_token = np.random.default_rng(22).integers(0, T, size=rows_max).astype(np.int32)
    W1 = _rand((S, d, f), 23, d ** -0.5)
    W3 = _rand((S, d, f), 24, d ** -0.5)
    W2 = _rand((S, f, d), 25, f ** -0.5)
    dev = torch.device("cuda")
    xg, rt = x.cuda(), torch.from_numpy(row_token).cuda()
    xp = xg[rt.long()].contiguous()
    offg = torch.from_numpy(off).cuda()
    W1g, W3g, W2g = W1.cuda(), W3.cuda(), W2.cuda()
    ws = torch.zeros(M.ffn_workspace_size(rows_max, f, "bf16"), dtype=torch.uint8, device=dev)
    cfg = M.make_config(T=T, d=d, N=S, f=f, k=1, dtype="bf16")
    copy = torch.full((rows_max, d), 7.0, dtype=torch.bfloat16, device=dev)
    M.moe_expert_ffn(cfg, xp, offg, S, rows_max, f, W1g, W3g, W2g, copy, ws)
    fused = torch.full((rows_max, d), 7.0, dtype=torch.bfloat16, device=dev)
    M.moe_expert_ffn_gather(cfg, xg, rt, offg, S, rows_max, f, W1g, W3g, W2g, fused, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    assert torch.equal(fused[:P], copy[:P])
    assert torch.all(fused[P:] == 7.0), "rows past the last segment were written"
    got = fused.float().cpu().numpy()
    xs = x[torch.from_numpy(row_token).long()]
    for s in range(S):
        a, b = int(off[s]), int(off[s + 1])
        if a < b:
            ref = O.swiglu(G.np32(xs[a:b]), G.np32(W1[s]), G.np32(W3[s]), G.np32(W2[s]), "bf16")
            G.assert_output_close(got[a:b], ref, "bf16", f"segment {s}")


def test_expert_ffn_gather_out_of_range_token_reads_zeros(gemm_form):
    """A row_token entry outside [0, T) is caught by the kernel's own bounds
    check: that row reads zeros (its output is exactly 0) and the status word
    records MOE_ERR_DEVICE_BOUNDS; every other row is unaffected."""
    sizes, d, f, T = [200, 90, 300], 256, 256, 400
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P
    x = _rand((T, d), 31)
    row_token = np.random.default_rng(32).integers(0, T, size=rows_max).astype(np.int32)
    bad = [5, 260, P - 1]
    row_token[bad] = [T, -3, 1 << 30]
    W1 = _rand((S, d, f), 33, d ** -0.5).cuda()
    W3 = _rand((S, d, f), 34, d ** -0.5).cuda()
    W2 = _rand((S, f, d), 35, f ** -0.5).cuda()
    dev = torch.device("cuda")
    xg = x.cuda()
    rt = torch.from_numpy(row_token).cuda()
    xp = xg[rt.clamp(0, T - 1).long()].contiguous()
    xp[bad] = 0
    offg = torch.from_numpy(off).cuda()
    cfg = M.make_config(T=T, d=d, N=S, f=f, k=1, dtype="bf16")
    ws = torch.zeros(M.ffn_workspace_size(rows_max, f, "bf16"), dtype=torch.uint8, device=dev)
    copy = torch.empty((rows_max, d), dtype=torch.bfloat16, device=dev)
    M.moe_expert_ffn(cfg, xp, offg, S, rows_max, f, W1, W3, W2, copy, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    fused = torch.empty_like(copy)
    M.moe_expert_ffn_gather(cfg, xg, rt, offg, S, rows_max, f, W1, W3, W2, fused, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_ERR_DEVICE_BOUNDS
    assert not fused[bad].any()
    assert torch.equal(fused, copy)
    M.moe_clear_device_status(ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK


def test_expert_ffn_on_a_slice_of_the_gpu():
    """moe_expert_ffn_on_sms: the same rows as moe_expert_ffn on any number of
    SMs, and a device group's call (offsets and weights pointing at its first
    expert) reproduces that group's rows of the whole-layer call."""
    sizes, d, f = [700, 0, 260, 1, 513, 90], 256, 384
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P + 3
    xp = _rand((rows_max, d), 13)
    W1 = _rand((S, d, f), 14, d ** -0.5)
    W3 = _rand((S, d, f), 15, d ** -0.5)
    W2 = _rand((S, f, d), 16, f ** -0.5)
    cfg = M.make_config(T=1, d=d, N=S, f=f, k=1, dtype="bf16")
    dev = torch.device("cuda")
    xg, W1g, W3g, W2g = xp.cuda(), W1.cuda(), W3.cuda(), W2.cuda()
    offg = torch.from_numpy(off).cuda()
    ws = torch.zeros(M.ffn_workspace_size(rows_max, f, "bf16"), dtype=torch.uint8, device=dev)
    full = torch.zeros((rows_max, d), dtype=torch.bfloat16, device=dev)
    M.moe_expert_ffn(cfg, xg, offg, S, rows_max, f, W1g, W3g, W2g, full, ws)
    for max_sms in (1, 2, 7, 18, 148, 1000):
        op = torch.zeros_like(full)
        M.moe_expert_ffn_on_sms(cfg, xg, offg, S, rows_max, f, W1g, W3g, W2g, op, max_sms, ws)
        torch.cuda.synchronize()
        assert M.moe_get_device_status(ws) == M.MOE_OK
        if max_sms >= 2:  # the same GEMM form: the same bits
            assert torch.equal(op, full), max_sms
        got = op.float().cpu().numpy()
        for s in range(S):
            a, b = int(off[s]), int(off[s + 1])
            if a < b:
                ref = O.swiglu(G.np32(xp[a:b]), G.np32(W1[s]), G.np32(W3[s]), G.np32(W2[s]), "bf16")
                G.assert_output_close(got[a:b], ref, "bf16", f"segment {s}, {max_sms} SMs")
    # experts 2..4 as one device on 18 SMs
    lo, hi = 2, 5
    op = torch.zeros_like(full)
    M.moe_expert_ffn_on_sms(cfg, xg, offg.data_ptr() + 4 * lo, hi - lo, rows_max, f,
                            W1g[lo].data_ptr(), W3g[lo].data_ptr(), W2g[lo].data_ptr(), op, 18, ws)
    torch.cuda.synchronize()
    a, b = int(off[lo]), int(off[hi])
    assert torch.equal(op[a:b], full[a:b])
    assert not op[:a].any() and not op[b:].any()


def _e4m3_codes(values) -> np.ndarray:
    """Byte codes of values that are e4m3 values (exact conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _a256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("sizes,d,f", [
    ([130, 0, 170, 1, 249], 256, 384),
    ([8, 8, 7, 9, 8, 8, 8, 8], 512, 1408),     # decode-like: a handful of rows per expert
    ([300, 400], 128, 256),
    ([600, 0, 513], 256, 512),                  # several 256-row pair tiles, ragged tails
])
def test_expert_ffn_e4m3_against_oracle(sizes, d, f, gemm_form):
    """FP8 experts (e4m3 x e4m3 on the tensor cores): the token rows' e4m3
    codes and row scales bit for bit against the oracle's quantization, and the
    output against the oracle's FP8 expert (weights dequantized, operand rows
    quantized per row) within the bf16 tolerance."""
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    rows_max = P + 5
    xp = _rand((rows_max, d), 21)
    Wb = {n: _rand(shape, seed, scale) for n, shape, seed, scale in (
        ("W1", (S, d, f), 22, d ** -0.5), ("W3", (S, d, f), 23, d ** -0.5),
        ("W2", (S, f, d), 24, f ** -0.5))}
    q = {}
    for n in Wb:  # per-column quantization, stored K-major
        qb, sc = W.quantize_e4m3(Wb[n])
        q[n] = (qb.transpose(-1, -2).contiguous(), sc)
    deq = {n: O.dequantize_e4m3(q[n][0].numpy(), q[n][1].numpy(), kmajor=True) for n in q}
    cfg = M.make_config(T=1, d=d, N=S, f=f, k=1, dtype="bf16")
    dev = torch.device("cuda")
    qd = {n: (q[n][0].cuda(), q[n][1].cuda()) for n in q}
    ex = M.e4m3_experts(qd["W1"][0], qd["W3"][0], qd["W2"][0], qd["W1"][1], qd["W3"][1],
                        qd["W2"][1])
    op = torch.zeros((rows_max, d), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(M.ffn_workspace_size_e4m3(rows_max, d, f), dtype=torch.uint8, device=dev)
    M.moe_expert_ffn_e4m3(cfg, xp.cuda(), torch.from_numpy(off).cuda(), S, rows_max, f, ex, op, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    # the workspace layout of moe_ffn_workspace_size_e4m3: control block, bf16
    # hidden rows, e4m3 token rows, their scales, ...
    o_xq = M.MOE_CTRL_BYTES + _a256(rows_max * f * 2)
    o_xs = o_xq + _a256(rows_max * d)
    w_h = ws.cpu().numpy()
    xq = w_h[o_xq:o_xq + P * d].reshape(P, d)
    xs = w_h[o_xs:o_xs + 4 * P].view(np.float32)
    vals, scale = O.quantize_rows_e4m3(G.np32(xp[:P]))
    assert np.array_equal(xs.view(np.uint32), scale.view(np.uint32)), "row scales differ"
    assert np.array_equal(xq, _e4m3_codes(vals)), "e4m3 codes of the token rows differ"
    got = op.float().cpu().numpy()
    for s in range(S):
        a, b = int(off[s]), int(off[s + 1])
        if a < b:
            ref = O.swiglu(G.np32(xp[a:b]), deq["W1"][s], deq["W3"][s], deq["W2"][s], "bf16",
                           act_e4m3=True)
            G.assert_output_close(got[a:b], ref, "bf16", f"segment {s}")
    assert not op[P:].any()


@pytest.mark.parametrize("sizes,d,f", [([100, 0, 37, 64], 128, 256), ([5], 64, 200)])
def test_expert_ffn_f32_against_oracle(sizes, d, f):
    S = len(sizes)
    off = _segments(sizes)
    P = int(off[-1])
    xp = _rand((P, d), 7, dtype=torch.float32)
    W1 = _rand((S, d, f), 8, d ** -0.5, torch.float32)
    W3 = _rand((S, d, f), 9, d ** -0.5, torch.float32)
    W2 = _rand((S, f, d), 10, f ** -0.5, torch.float32)
    cfg = M.make_config(T=1, d=d, N=S, f=f, k=1, dtype="f32")
    dev = torch.device("cuda")
    op = torch.zeros((P, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(M.ffn_workspace_size(P, f, "f32"), dtype=torch.uint8, device=dev)
    M.moe_expert_ffn(cfg, xp.cuda(), torch.from_numpy(off).cuda(), S, P, f, W1.cuda(), W3.cuda(),
                     W2.cuda(), op, ws)
    torch.cuda.synchronize()
    got = op.cpu().numpy()
    for s in range(S):
        a, b = int(off[s]), int(off[s + 1])
        if a == b:
            continue
        ref = O.swiglu(xp[a:b].numpy(), W1[s].numpy(), W3[s].numpy(), W2[s].numpy(), "f32")
        G.assert_output_close(got[a:b], ref, "f32", f"segment {s}")


def test_transposed_tails_equal_padded_bit_for_bit(monkeypatch):
    """Tiles computed transposed (the default in pair form: every segment's
    last tile, and every tile of the second GEMM and of the plain grouped
    GEMM) give the same bits as the untransposed form with the tails padded
    to 256 rows (MOE_GEMM_SWAP_TAILS=0): each output is the same sum over the
    same k."""
    monkeypatch.setenv("MOE_GEMM_CTA_PAIRS", "1")
    sizes, d, f = TAIL_SIZES, 320, 192
    S = len(sizes)
    off = torch.from_numpy(_segments(sizes)).cuda()
    rows_max = int(sum(sizes)) + 5
    dev = torch.device("cuda")
    xp = _rand((rows_max, d), 51).cuda()
    W1 = _rand((S, d, f), 52, d ** -0.5).cuda()
    W3 = _rand((S, d, f), 53, d ** -0.5).cuda()
    W2 = _rand((S, f, d), 54, f ** -0.5).cuda()
    B = _rand((S, d, 320), 55, d ** -0.5).cuda()
    cfg = M.make_config(T=1, d=d, N=S, f=f, k=1, dtype="bf16")
    outs = []
    for swap in ("1", "0"):
        monkeypatch.setenv("MOE_GEMM_SWAP_TAILS", swap)
        op = torch.zeros((rows_max, d), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(M.ffn_workspace_size(rows_max, f, "bf16"), dtype=torch.uint8, device=dev)
        M.moe_expert_ffn(cfg, xp, off, S, rows_max, f, W1, W3, W2, op, ws)
        g = torch.zeros((rows_max, 320), dtype=torch.bfloat16, device=dev)
        M.moe_grouped_gemm("bf16", xp, off, S, rows_max, d, 320, B, g, ws)
        torch.cuda.synchronize()
        assert M.moe_get_device_status(ws) == M.MOE_OK
        outs.append((op.cpu(), g.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]), "expert FFN: transposed and padded tails differ"
    assert torch.equal(outs[0][1], outs[1][1]), "grouped GEMM: transposed and padded tails differ"
