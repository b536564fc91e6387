"""Seeded synthetic workloads for the sparse MoE FFN layer.

This module only draws inputs. It holds none of the layer's arithmetic, so the
CPU oracle (``oracle/``) and the CUDA library can both be fed from it without
sharing any code path.

Recipe (one fixed draw order per workload, ``torch.Generator().manual_seed``):
  x    ~ N(0, 1)            [T, d]
  W_r  ~ N(0, 1/d)          [d, N]      router ("Understanding Mixture of
                                          Experts", §"Expert and Router")
  W1   ~ N(0, 1/d)          [N, d, f]   SwiGLU gate projection
  W3   ~ N(0, 1/d)          [N, d, f]   SwiGLU up projection
  W2   ~ N(0, 1/f)          [N, f, d]   SwiGLU down projection
  Ws1, Ws3 ~ N(0, 1/d)      [d, fs]     shared expert ("How to design inference
  Ws2  ~ N(0, 1/fs)         [fs, d]      cost with MoE routing", §"how routing
                                          allocates the compute budget")
Values are drawn in fp32; bf16 workloads round each value once to bf16
(round-to-nearest-even). Workloads with e4m3 routed experts quantize W1, W3
and W2 per output column (quantize_e4m3) and store the bytes K-major,
W1q [N, f, d], W3q [N, f, d], W2q [N, d, f], with scales [N, f] and [N, d].
The optional router bias is the log of a Zipf(s) distribution over experts, expert 0 the most popular, to skew the load the way
the straggler discussion of "Capacity-Aware Inference: Mitigating the
Straggler Effect in MoE" (§1) describes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

TOKEN_CHOICE = "token_choice"
EXPERT_CHOICE = "expert_choice"
CAPACITY_DROP = "capacity_drop"
CAPACITY_DROP_DEVICE = "capacity_drop_device"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    N: int
    f: int
    k: int
    mode: str = TOKEN_CHOICE
    gamma: float = math.inf
    m: int = 0
    group_size: int = 8
    renorm: bool = False
    f_shared: int = 0
    dtype: str = "bf16"          # "bf16" or "f32": activations, weights, output
    weights: str = "same"        # "same" (the dtype) or "e4m3": routed experts in FP8
    zipf_s: Optional[float] = None
    seed: int = 0

    @property
    def kc(self) -> int:
        """Candidate slots per token (expert choice: every expert)."""
        return self.N if self.mode == EXPERT_CHOICE else self.k + self.m

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def describe(self) -> str:
        s = (f"{self.name}: T={self.T} d={self.d} N={self.N} f={self.f} k={self.k} "
             f"mode={self.mode} dtype={self.dtype}")
        if self.mode == CAPACITY_DROP:
            s += f" gamma={self.gamma}"
        if self.mode == CAPACITY_DROP_DEVICE:
            s += f" gamma={self.gamma} device={self.group_size} experts"
        if self.m:
            s += f" expanded m={self.m} group={self.group_size}"
        if self.renorm:
            s += " renorm"
        if self.f_shared:
            s += f" shared f={self.f_shared}"
        if self.zipf_s is not None:
            s += f" zipf_s={self.zipf_s}"
        if self.weights == "e4m3":
            s += " routed experts in e4m3 (weights per-column, activations per-row scales)"
        return s


# The five workloads of the layer benchmark.
TINY_F32 = Workload("tiny_fp32", T=256, d=128, N=8, f=256, k=2, dtype="f32")
EC_BF16 = Workload("expert_choice_bf16", T=2048, d=1024, N=16, f=2816, k=2,
                   mode=EXPERT_CHOICE)
MIXTRAL_BF16 = Workload("mixtral_bf16", T=4096, d=4096, N=8, f=14336, k=2,
                        renorm=True, zipf_s=1.2)
FINE_BF16 = Workload("finegrained_bf16", T=8192, d=2048, N=64, f=1408, k=6,
                     mode=CAPACITY_DROP, gamma=1.25, f_shared=2816, zipf_s=1.0)
DECODE_BF16 = Workload("decode_bf16", T=32, d=4096, N=8, f=14336, k=2)
# the decode step with its routed experts in FP8 (e4m3 weights and activations)
DECODE_W8 = DECODE_BF16.replace(name="decode_e4m3", weights="e4m3")


def mixtral(gamma: float) -> Workload:
    """Mixtral-shaped layer at capacity factor gamma (inf = no capacity limit)."""
    if math.isinf(gamma):
        return MIXTRAL_BF16
    return MIXTRAL_BF16.replace(name=f"mixtral_bf16_gamma{gamma:g}",
                                mode=CAPACITY_DROP, gamma=gamma)


def fine_expanded() -> Workload:
    return FINE_BF16.replace(name="finegrained_bf16_expanded", m=4, group_size=8)


def fine_device() -> Workload:
    """The fine-grained layer with device-level capacity: 8 devices of 8
    experts, each holding 8 x 960 = 7680 candidates."""
    return FINE_BF16.replace(name="finegrained_bf16_device", mode=CAPACITY_DROP_DEVICE,
                             group_size=8)


ALL = {w.name: w for w in (TINY_F32, EC_BF16, MIXTRAL_BF16, mixtral(1.0), mixtral(1.5),
                           FINE_BF16, fine_expanded(), fine_device(), DECODE_BF16, DECODE_W8)}


def zipf_log_probs(N: int, s: float) -> np.ndarray:
    """Router bias b_e = ln p_e with p_e = (e+1)^-s / sum_j (j+1)^-s, in fp64, rounded to fp32."""
    w = np.array([(e + 1.0) ** (-s) for e in range(N)], dtype=np.float64)
    return np.log(w / w.sum()).astype(np.float32)


def _draw(g: torch.Generator, shape, std: float) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def make_inputs(w: Workload, with_experts: bool = True) -> Dict[str, torch.Tensor]:
    """Draw the workload's inputs on the CPU.

    Returns torch CPU tensors in the workload dtype (bf16 or fp32), plus an fp32
    ``bias`` (or None). ``with_experts=False`` stops after the router weights,
    for routing-only tests; the x and W_r values are the same either way.
    """
    g = torch.Generator().manual_seed(w.seed)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _draw(g, (w.T, w.d), 1.0).to(dt)
    out["W_r"] = _draw(g, (w.d, w.N), w.d ** -0.5).to(dt)
    out["bias"] = (torch.from_numpy(zipf_log_probs(w.N, w.zipf_s))
                   if w.zipf_s is not None else None)
    if not with_experts:
        return out
    out["W1"] = _draw(g, (w.N, w.d, w.f), w.d ** -0.5).to(dt)
    out["W3"] = _draw(g, (w.N, w.d, w.f), w.d ** -0.5).to(dt)
    out["W2"] = _draw(g, (w.N, w.f, w.d), w.f ** -0.5).to(dt)
    if w.weights == "e4m3":  # stored K-major: [N, n, K] bytes, [N, n] scales
        for name in ("W1", "W3", "W2"):
            q, sc = quantize_e4m3(out[name])
            out[name + "q"], out[name + "s"] = q.transpose(-1, -2).contiguous(), sc
    if w.f_shared:
        fs = w.f_shared
        out["Ws1"] = _draw(g, (w.d, fs), w.d ** -0.5).to(dt)
        out["Ws3"] = _draw(g, (w.d, fs), w.d ** -0.5).to(dt)
        out["Ws2"] = _draw(g, (fs, w.d), fs ** -0.5).to(dt)
    else:
        out["Ws1"] = out["Ws3"] = out["Ws2"] = None
    return out


E4M3_MAX = 448.0


def quantize_e4m3(W: torch.Tensor):
    """Weights [..., K, n] -> (bytes [..., K, n] uint8, scale [..., n] fp32):
    per output column, scale = max_k |W| / 448 (1 for an all-zero column) and
    each weight is W / scale rounded to the nearest e4m3 value (ties to even,
    the magnitude clamped to 448), so that W ~ value(byte) * scale."""
    Wf = W.float()
    amax = Wf.abs().amax(dim=-2)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (Wf / scale.unsqueeze(-2)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def random_logits(T: int, N: int, seed: int, scale: float = 1.0,
                  quantum: Optional[float] = None) -> torch.Tensor:
    """fp32 router logits for routing-only cases. ``quantum`` snaps values to a
    grid so that ties (equal logits within a token and equal gates across
    tokens) occur often."""
    g = torch.Generator().manual_seed(seed)
    L = torch.randn((T, N), generator=g, dtype=torch.float32) * scale
    if quantum is not None:
        L = torch.round(L / quantum) * quantum
    return L


def to_numpy_f32(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact widening of a bf16/fp32 tensor to an fp32 numpy array."""
    if t is None:
        return None
    return t.float().numpy()
