"""Seeded synthetic inputs for KDA workloads.

This module only draws random tensors. It holds none of KDA's arithmetic and
imports neither the device library nor the oracle; the tests hand the same
tensors to both sides.

Recipe (all draws in fp32, then cast with round-to-nearest-even):
  q, k       ~ N(0, 1), each token-head row scaled to unit L2 norm
  v          ~ N(0, 1)
  beta       = sigmoid(N(0, 1)), one per token and head
  log_alpha  = max(-exp(N(-3, 1)), log 0.5), one per token, head and key channel
               (the retention lower bound of 0.5; see the K3 training overview,
               zuoshipin.com/article/18261, sections 2 and 6, which bound the
               per-step retention from below but give no value)
  gate       = sigmoid(N(0, 1)) over value channels
  S0         ~ N(0, 0.1^2) where a workload starts from a non-zero state

Each tensor has its own stream: a torch generator on the target device seeded
from (seed, tensor id, step). Ids: q=0, k=1, v=2, beta=3, log_alpha=4, gate=5,
S0=6.

Workloads (the pages give no head counts or widths for KDA; these are chosen
shapes, with the 1,048,576-token context the K3 pages quote as the model's
maximum, K3 explainer, devpress.csdn.net, section 1):
  tiny     1 x 256 tokens, H=2, d=64, fp32, zero initial state
  prefill  4 x 4096 tokens, H=16, d=128, bf16, S0 ~ N(0, 0.01)
  varlen   8 packed sequences, lengths uniform in [1024, 32768] (PCG64 seed 2),
           H=32, d=128, bf16, zero initial state
  longctx  1 x 1,048,576 tokens, H=16, d=128, bf16, 8 segments of 131,072
  decode   256 sequences x H=32, d=128, one bf16 token per step, 64 steps,
           fp32 state ~ N(0, 0.01)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "beta": 3, "log_alpha": 4, "gate": 5, "S0": 6}
LOG_ALPHA_FLOOR = math.log(0.5)


@dataclass
class Workload:
    name: str
    lengths: list
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    seed: int
    init_state: bool
    n_segments: int = 0
    steps: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def T_total(self) -> int:
        return int(sum(self.lengths))

    @property
    def cu_seqlens(self) -> list:
        return [0] + list(np.cumsum(self.lengths, dtype=np.int64).tolist())


def varlen_lengths(seed: int = 2, n: int = 8, lo: int = 1024, hi: int = 32768):
    """Sequence lengths drawn uniformly from [lo, hi] with a fixed seed."""
    return [int(x) for x in np.random.Generator(np.random.PCG64(seed)).integers(lo, hi + 1, n)]


WORKLOADS = {
    "tiny": Workload("tiny", [256], 2, 64, 64, torch.float32, 0, False),
    "prefill": Workload("prefill", [4096] * 4, 16, 128, 128, torch.bfloat16, 1, True),
    "varlen": Workload("varlen", varlen_lengths(), 32, 128, 128, torch.bfloat16, 2, False),
    "longctx": Workload("longctx", [1 << 20], 16, 128, 128, torch.bfloat16, 3, False,
                        n_segments=8),
    "decode": Workload("decode", [1] * 256, 32, 128, 128, torch.bfloat16, 4, True, steps=64),
}


def _gen(seed: int, tensor: str, step: int, device) -> torch.Generator:
    s = np.random.SeedSequence([int(seed), TENSOR_IDS[tensor], int(step)])
    g = torch.Generator(device=device)
    g.manual_seed(int(s.generate_state(1, np.uint64)[0]) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _randn(shape, seed, tensor, step, device):
    return torch.randn(shape, generator=_gen(seed, tensor, step, device),
                       device=device, dtype=torch.float32)


def _unit_rows(x):
    return x / torch.sqrt(torch.sum(x * x, dim=-1, keepdim=True))


def tokens(n_tokens: int, H: int, dk: int, dv: int, dtype=torch.bfloat16, seed: int = 0,
           step: int = 0, device="cpu", with_gate: bool = True) -> dict:
    """Per-token inputs q, k, v, beta, log_alpha, gate (None if not with_gate)."""
    dev = torch.device(device)
    q = _unit_rows(_randn((n_tokens, H, dk), seed, "q", step, dev)).to(dtype)
    k = _unit_rows(_randn((n_tokens, H, dk), seed, "k", step, dev)).to(dtype)
    v = _randn((n_tokens, H, dv), seed, "v", step, dev).to(dtype)
    beta = torch.sigmoid(_randn((n_tokens, H), seed, "beta", step, dev)).to(dtype)
    la = -torch.exp(_randn((n_tokens, H, dk), seed, "log_alpha", step, dev) - 3.0)
    la = torch.clamp_min(la, LOG_ALPHA_FLOOR).to(dtype)
    g = None
    if with_gate:
        g = torch.sigmoid(_randn((n_tokens, H, dv), seed, "gate", step, dev)).to(dtype)
    return {"q": q, "k": k, "v": v, "beta": beta, "log_alpha": la, "gate": g}


def state(n: int, H: int, dk: int, dv: int, seed: int = 0, device="cpu", std: float = 0.1):
    """fp32 state [n, H, dk, dv] ~ N(0, std^2)."""
    return _randn((n, H, dk, dv), seed, "S0", 0, torch.device(device)) * std


def make(workload: str | Workload, device="cpu", step: int = 0, n_tokens: int | None = None):
    """All inputs of a prefill-style workload: tokens + cu_seqlens + S0."""
    w = WORKLOADS[workload] if isinstance(workload, str) else workload
    T = w.T_total if n_tokens is None else n_tokens
    d = tokens(T, w.H, w.dk, w.dv, w.dtype, w.seed, step, device)
    d["cu_seqlens"] = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=device)
    n_seq = len(w.lengths)
    d["S0"] = state(n_seq, w.H, w.dk, w.dv, w.seed, device) if w.init_state else None
    return d
