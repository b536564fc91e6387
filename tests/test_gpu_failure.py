"""Failure detection on the GPU without a GPU fault: a bounded wait that
runs out returns an error status the host reads, and the context stays
usable (the self-test withholds one k-block of the tensor-core GEMM)."""
import pytest
import torch

import routing_capacity_drop_router_b300 as M

pytestmark = pytest.mark.gpu


def _gemm_inputs(S=2, rows_per=200, K=256, n_out=384):
    g = torch.Generator().manual_seed(11)
    rows = S * rows_per
    A = (torch.randn(rows, K, generator=g) * 0.5).to(torch.bfloat16).cuda()
    B = (torch.randn(S, K, n_out, generator=g) / K ** 0.5).to(torch.bfloat16).cuda()
    offs = torch.arange(0, rows + 1, rows_per, dtype=torch.int32).cuda()
    out = torch.zeros(rows, n_out, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(M.ffn_workspace_size(0, 0, "bf16"), dtype=torch.uint8, device="cuda")
    return A, B, offs, out, ws, S, rows, K, n_out


@pytest.mark.parametrize("pairs", ["1", "0"], ids=["cta_pairs", "single_cta"])
def test_expired_wait_reports_timeout_and_context_survives(pairs, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_CTA_PAIRS", pairs)
    A, B, offs, out, ws, S, rows, K, n_out = _gemm_inputs()
    M.moe_selftest_expired_wait(A, offs, S, rows, K, n_out, B, out, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_ERR_DEVICE_TIMEOUT
    # the same workspace and context keep working once the status is cleared
    M.moe_clear_device_status(ws)
    out.zero_()
    M.moe_grouped_gemm("bf16", A, offs, S, rows, K, n_out, B, out, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == M.MOE_OK
    rp = rows // S
    ref = torch.cat([A[i * rp:(i + 1) * rp].float() @ B[i].float() for i in range(S)])
    err = (out.float() - ref).norm() / ref.norm()
    assert err < 1e-2, float(err)
