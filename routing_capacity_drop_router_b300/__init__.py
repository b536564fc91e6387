"""Python binding of the B300 sparse MoE FFN layer library (``libmoe_b300.so``).

Argument marshalling only: every function here forwards torch CUDA tensors
(device pointers) and the current CUDA stream to the C entry point of the
same name declared in ``include/moe.h``, and raises ``MoeError`` on a
non-zero status. All arithmetic runs in the library's CUDA kernels; there is
no CPU path. The library is built in-tree with
``python -m routing_capacity_drop_router_b300.build``.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_NULL = -1
MOE_ERR_SHAPE = -2
MOE_ERR_ALIGN = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_UNSUPPORTED = -5
MOE_ERR_LAUNCH = -6
MOE_ERR_DEVICE_TIMEOUT = -7
MOE_ERR_DEVICE_BOUNDS = -8

MOE_TOKEN_CHOICE = 0
MOE_EXPERT_CHOICE = 1
MOE_CAPACITY_DROP = 2
MOE_CAPACITY_DROP_DEVICE = 3
MOE_F32 = 0
MOE_BF16 = 1
MOE_LOGITS_GIVEN = 1
MOE_FUSE_GATHER = 2
MOE_STATS_LEN = 8
MOE_CTRL_BYTES = 1024
MOE_NOALLOC_SCRATCH_BYTES = 64 << 20

MODES = {"token_choice": MOE_TOKEN_CHOICE, "expert_choice": MOE_EXPERT_CHOICE,
         "capacity_drop": MOE_CAPACITY_DROP, "capacity_drop_device": MOE_CAPACITY_DROP_DEVICE}
DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("N", ctypes.c_int32),
                ("f", ctypes.c_int32), ("k", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("gamma", ctypes.c_double), ("m", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("f_shared", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class moe_sizes_t(ctypes.Structure):
    _fields_ = [("kc", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("rows_max", ctypes.c_int64), ("workspace", ctypes.c_size_t),
                ("ffn_workspace", ctypes.c_size_t)]


class moe_e4m3_experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W1", "W3", "W2", "s1", "s3", "s2")]


class moe_views_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "status", "logits", "scores", "cand_idx", "cand_gate", "slot", "keep", "demand", "kept",
        "expert_offsets", "row_token", "row_gate", "tok_rows", "xp", "op", "shared_out",
        "coverage")]


# name -> (restype, argtypes)
_VP = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config)
SIGNATURES = {
    "moe_sizes": (ctypes.c_int, [_CFG, ctypes.POINTER(moe_sizes_t)]),
    "moe_workspace_size": (ctypes.c_size_t, [_CFG]),
    "moe_ffn_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    "moe_route_workspace_size": (ctypes.c_size_t, [_CFG]),
    "moe_ffn_workspace_size_e4m3": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32,
                                                      ctypes.c_int32]),
    "moe_workspace_size_e4m3": (ctypes.c_size_t, [_CFG]),
    "moe_route": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                 ctypes.c_size_t, _VP]),
    "moe_capacity_drop": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_dispatch": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                    _VP]),
    "moe_expert_ffn": (ctypes.c_int, [_CFG, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                      ctypes.c_int32, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t,
                                      _VP]),
    "moe_expert_ffn_noalloc": (ctypes.c_int, [_CFG, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_int32, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_expert_ffn_gather": (ctypes.c_int, [_CFG, _VP, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.c_int32, _VP, _VP, _VP, _VP, _VP,
                                             ctypes.c_size_t, _VP]),
    "moe_expert_ffn_on_sms": (ctypes.c_int, [_CFG, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.c_int32, _VP, _VP, _VP, _VP, ctypes.c_int32,
                                             _VP, ctypes.c_size_t, _VP]),
    "moe_expert_ffn_e4m3": (ctypes.c_int, [_CFG, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_int32, ctypes.c_void_p, _VP, _VP,
                                           ctypes.c_size_t, _VP]),
    "moe_layer_forward_e4m3": (ctypes.c_int, [_CFG, _VP, _VP, _VP, ctypes.c_void_p, _VP, _VP,
                                              _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t,
                                              _VP]),
    "moe_grouped_gemm": (ctypes.c_int, [ctypes.c_int32, _VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                        ctypes.c_int32, ctypes.c_int32, _VP, _VP, _VP,
                                        ctypes.c_size_t, _VP]),
    "moe_selftest_expired_wait": (ctypes.c_int, [_VP, _VP, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.c_int32, _VP, _VP, _VP,
                                                 ctypes.c_size_t, _VP]),
    "moe_combine": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_load_stats": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "moe_layer_forward": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                         _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "moe_workspace_views": (ctypes.c_int, [_CFG, _VP, ctypes.POINTER(moe_views_t)]),
    "moe_layer_stages": (ctypes.c_int, [_CFG, ctypes.POINTER(ctypes.c_char_p), ctypes.c_int]),
    "moe_set_trace_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    "moe_get_device_status": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(ctypes.c_int32)]),
    "moe_clear_device_status": (ctypes.c_int, [_VP, _VP]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_release_caches": (None, []),
}

_lib_handle = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m routing_capacity_drop_router_b300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def make_config(*, T: int, d: int, N: int, f: int, k: int, mode="token_choice",
                gamma: float = math.inf, m: int = 0, group_size: int = 8, renorm: bool = False,
                f_shared: int = 0, dtype="bf16", logits_given: bool = False,
                fuse_gather: bool = False) -> moe_config:
    return moe_config(T=T, d=d, N=N, f=f, k=k, mode=MODES.get(mode, mode), gamma=float(gamma),
                      m=m, group_size=group_size, renorm=int(bool(renorm)), f_shared=f_shared,
                      dtype=DTYPES.get(dtype, dtype),
                      flags=(MOE_LOGITS_GIVEN if logits_given else 0) |
                      (MOE_FUSE_GATHER if fuse_gather else 0))


def config_from_workload(w, logits_given: bool = False, fuse_gather: bool = False) -> moe_config:
    """moe_config from any object with the workload fields (T, d, N, f, k,
    mode, gamma, m, group_size, renorm, f_shared, dtype)."""
    return make_config(T=w.T, d=w.d, N=w.N, f=w.f, k=w.k, mode=w.mode, gamma=w.gamma, m=w.m,
                       group_size=w.group_size, renorm=w.renorm, f_shared=w.f_shared,
                       dtype=w.dtype, logits_given=logits_given, fuse_gather=fuse_gather)


def _p(t) -> Optional[int]:
    """Device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def sizes(cfg: moe_config) -> moe_sizes_t:
    out = moe_sizes_t()
    _check(lib().moe_sizes(ctypes.byref(cfg), ctypes.byref(out)), "moe_sizes")
    return out


def workspace_size(cfg: moe_config) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg)))


def ffn_workspace_size(rows_max: int, f: int, dtype) -> int:
    return int(lib().moe_ffn_workspace_size(rows_max, f, DTYPES.get(dtype, dtype)))


def ffn_workspace_size_e4m3(rows_max: int, d: int, f: int) -> int:
    return int(lib().moe_ffn_workspace_size_e4m3(rows_max, d, f))


def workspace_size_e4m3(cfg: moe_config) -> int:
    return int(lib().moe_workspace_size_e4m3(ctypes.byref(cfg)))


def route_workspace_size(cfg: moe_config) -> int:
    return int(lib().moe_route_workspace_size(ctypes.byref(cfg)))


def moe_route(cfg, x, W_router, bias, logits, scores, cand_idx, cand_gate, ws, home_group=None,
              stream=None) -> None:
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(W_router), _p(bias), _p(logits),
                           _p(scores), _p(cand_idx), _p(cand_gate), _p(home_group), _p(ws),
                           ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def moe_capacity_drop(cfg, cand_idx, cand_gate, slot, keep, demand, kept, stream=None) -> None:
    _check(lib().moe_capacity_drop(ctypes.byref(cfg), _p(cand_idx), _p(cand_gate), _p(slot),
                                   _p(keep), _p(demand), _p(kept), _stream(stream)),
           "moe_capacity_drop")


def moe_dispatch(cfg, x, cand_idx, cand_gate, slot, kept, expert_offsets, row_token, row_gate,
                 tok_rows, xp, coverage=None, stream=None) -> None:
    _check(lib().moe_dispatch(ctypes.byref(cfg), _p(x), _p(cand_idx), _p(cand_gate), _p(slot),
                              _p(kept), _p(expert_offsets), _p(row_token), _p(row_gate),
                              _p(tok_rows), _p(coverage), _p(xp), _stream(stream)),
           "moe_dispatch")


def moe_expert_ffn(cfg, xp, offsets, n_segments, rows_max, f, W1, W3, W2, op, ws,
                   stream=None) -> None:
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _p(xp), _p(offsets), n_segments, rows_max, f,
                                _p(W1), _p(W3), _p(W2), _p(op), _p(ws), ws.numel() * ws.element_size(),
                                _stream(stream)), "moe_expert_ffn")


def e4m3_experts(W1q, W3q, W2q, s1, s3, s2) -> moe_e4m3_experts:
    """The pointer struct of e4m3 routed experts (tensors must stay alive)."""
    return moe_e4m3_experts(*(_p(t) for t in (W1q, W3q, W2q, s1, s3, s2)))


def moe_expert_ffn_e4m3(cfg, xp, offsets, n_segments, rows_max, f, experts, op, ws,
                        stream=None) -> None:
    _check(lib().moe_expert_ffn_e4m3(ctypes.byref(cfg), _p(xp), _p(offsets), n_segments, rows_max,
                                     f, ctypes.byref(experts), _p(op), _p(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_e4m3")


def moe_expert_ffn_gather(cfg, x, row_token, offsets, n_segments, rows_max, f, W1, W3, W2, op, ws,
                          stream=None) -> None:
    """moe_expert_ffn whose first GEMM reads row r from x[row_token[r]] (bf16)."""
    _check(lib().moe_expert_ffn_gather(ctypes.byref(cfg), _p(x), _p(row_token), _p(offsets),
                                       n_segments, rows_max, f, _p(W1), _p(W3), _p(W2), _p(op),
                                       _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_gather")


def moe_expert_ffn_on_sms(cfg, xp, offsets, n_segments, rows_max, f, W1, W3, W2, op, max_sms, ws,
                          stream=None) -> None:
    """moe_expert_ffn on at most ``max_sms`` SMs (bf16). ``offsets``, ``W1``,
    ``W3``, ``W2`` may be raw device addresses (int) into larger arrays."""
    _check(lib().moe_expert_ffn_on_sms(ctypes.byref(cfg), _p(xp), _p(offsets), n_segments,
                                       rows_max, f, _p(W1), _p(W3), _p(W2), _p(op), max_sms,
                                       _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_on_sms")


def moe_expert_ffn_noalloc(cfg, xp, offsets, n_segments, rows_max, f, W1, W3, W2, op,
                           device_status=None, stream=None) -> None:
    """moe_expert_ffn without a workspace, for callers that cannot allocate
    device memory (the library keeps the hidden activations in its own
    MOE_NOALLOC_SCRATCH_BYTES device array; calls that overlap on the GPU
    race on it)."""
    _check(lib().moe_expert_ffn_noalloc(ctypes.byref(cfg), _p(xp), _p(offsets), n_segments,
                                        rows_max, f, _p(W1), _p(W3), _p(W2), _p(op),
                                        _p(device_status), _stream(stream)),
           "moe_expert_ffn_noalloc")


def moe_grouped_gemm(dtype, A, offsets, n_segments, rows_max, K, n_out, B, out, ws,
                     stream=None) -> None:
    _check(lib().moe_grouped_gemm(DTYPES.get(dtype, dtype), _p(A), _p(offsets), n_segments,
                                  rows_max, K, n_out, _p(B), _p(out), _p(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_gemm")


def moe_selftest_expired_wait(A, offsets, n_segments, rows_max, K, n_out, B, out, ws,
                              stream=None) -> None:
    """Enqueue the bf16 grouped GEMM with one withheld k-block, so that its
    bounded wait expires and MOE_ERR_DEVICE_TIMEOUT lands in ws's status word
    (failure-detection self-test)."""
    _check(lib().moe_selftest_expired_wait(_p(A), _p(offsets), n_segments, rows_max, K, n_out,
                                           _p(B), _p(out), _p(ws),
                                           ws.numel() * ws.element_size(), _stream(stream)),
           "moe_selftest_expired_wait")


def moe_combine(cfg, op, row_gate, tok_rows, shared_out, y, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(cfg), _p(op), _p(row_gate), _p(tok_rows),
                             _p(shared_out), _p(y), _stream(stream)), "moe_combine")


def moe_load_stats(cfg, demand, kept, scores, stats, ws, stream=None) -> None:
    _check(lib().moe_load_stats(ctypes.byref(cfg), _p(demand), _p(kept), _p(scores), _p(stats),
                                _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_load_stats")


def moe_layer_forward(cfg, x, W_router, bias, W1, W3, W2, Ws1, Ws3, Ws2, y, ws, *,
                      home_group=None, logits=None, stats=None, stream=None) -> None:
    _check(lib().moe_layer_forward(ctypes.byref(cfg), _p(x), _p(W_router), _p(bias), _p(W1),
                                   _p(W3), _p(W2), _p(Ws1), _p(Ws3), _p(Ws2), _p(home_group),
                                   _p(logits), _p(y), _p(stats), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_layer_forward_e4m3(cfg, x, W_router, bias, experts, Ws1, Ws3, Ws2, y, ws, *,
                           home_group=None, logits=None, stats=None, stream=None) -> None:
    """moe_layer_forward with e4m3 routed experts (``experts`` from e4m3_experts)."""
    _check(lib().moe_layer_forward_e4m3(ctypes.byref(cfg), _p(x), _p(W_router), _p(bias),
                                        ctypes.byref(experts), _p(Ws1), _p(Ws3), _p(Ws2),
                                        _p(home_group), _p(logits), _p(y), _p(stats), _p(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_forward_e4m3")


def moe_workspace_views(cfg, ws) -> moe_views_t:
    out = moe_views_t()
    _check(lib().moe_workspace_views(ctypes.byref(cfg), _p(ws), ctypes.byref(out)),
           "moe_workspace_views")
    return out


def moe_layer_stages(cfg):
    """Names of the kernels moe_layer_forward launches for cfg, in order."""
    n = lib().moe_layer_stages(ctypes.byref(cfg), None, 0)
    if n < 0:
        raise MoeError(n, "moe_layer_stages")
    names = (ctypes.c_char_p * max(n, 1))()
    lib().moe_layer_stages(ctypes.byref(cfg), names, n)
    return [names[i].decode() for i in range(n)]


def moe_set_trace_events(events) -> None:
    """Record ``events`` (torch.cuda.Event with enable_timing, one more than
    the stages; ``None`` entries record nothing at that boundary) inside every
    later moe_layer_forward of this host thread; ``None`` or ``[]`` turns
    tracing off. Each event must have been created (recorded once) so that it
    has a CUDA handle."""
    events = list(events or [])
    handles = (ctypes.c_void_p * max(len(events), 1))()
    for i, ev in enumerate(events):
        if ev is None:
            continue  # no event at this stage boundary
        h = ev if isinstance(ev, int) else ev.cuda_event
        if not h:
            raise ValueError("event has no CUDA handle yet: record it once first")
        handles[i] = h
    _check(lib().moe_set_trace_events(handles, len(events)), "moe_set_trace_events")


def moe_get_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib().moe_get_device_status(_p(ws), _stream(stream), ctypes.byref(v)),
           "moe_get_device_status")
    return int(v.value)


def moe_clear_device_status(ws, stream=None) -> None:
    _check(lib().moe_clear_device_status(_p(ws), _stream(stream)), "moe_clear_device_status")


def view_tensor(ptr: int, shape, dtype, device=None):
    """A torch tensor aliasing device memory at ``ptr`` (a pointer from
    moe_workspace_views); valid while the workspace it points into lives."""
    import torch
    typestr = {torch.float32: "<f4", torch.int32: "<i4", torch.uint8: "|u1",
               torch.float64: "<f8", torch.bfloat16: "<i2"}[dtype]
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())

    class _Holder:
        __cuda_array_interface__ = {"shape": tuple(int(s) for s in shape), "typestr": typestr,
                                    "data": (int(ptr), False), "version": 3, "strides": None}

    t = torch.as_tensor(_Holder(), device=device)
    return t.view(torch.bfloat16) if dtype == torch.bfloat16 else t
