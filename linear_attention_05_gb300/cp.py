"""Context-parallel KDA over several ranks (one segment of one long sequence each).

K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context
parallel": every device processes its own segment and emits two fixed-size
pieces, how the segment rewrites the memory it is handed (the transition X,
dk x dk per head) and the state it builds from empty memory (Z, dk x dv per
head). Merging these in order with a prefix scan recovers the exact state
entering every segment, after which each device finishes its segment from that
state. The only exchange is one all-gather of H * (dk*dk + dk*dv) fp32 values
per rank (2 MiB at H = 16, d = 128); no key/value exchange is needed.

The three compute steps default to the library's entry points
(kda_segment_summary, kda_scan_combine, kda_chunk_fwd); they are parameters so
that the exchange logic can also be driven by other implementations.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _default_summary(k, v, log_alpha, beta, l2norm):
    from . import binding
    cu = torch.tensor([0, k.shape[0]], dtype=torch.int32, device=k.device)
    return binding.segment_summary(k, v, log_alpha, beta, cu, l2norm=l2norm)


def _default_scan(X, Z, S_init):
    from . import binding
    return binding.scan_combine(X, Z, S_init)


def _default_forward(q, k, v, log_alpha, beta, gate, entry, scale, l2norm):
    from . import binding
    out, fs = binding.chunk_fwd(q, k, v, log_alpha, beta, gate, entry[None].contiguous(), None,
                                n_seq=1, scale=scale, l2norm=l2norm)
    return out, fs[0]


def context_parallel_forward(q, k, v, log_alpha, beta, gate=None, initial_state=None,
                             group=None, scale=1.0, l2norm=True, summary=None, scan=None,
                             forward=None):
    """KDA over a sequence split across the ranks of `group`, rank r holding segment r.

    q, k, log_alpha: [T_r, H, dk]; v, gate: [T_r, H, dv]; beta: [T_r, H] (this rank's tokens)
    initial_state: [H, dk, dv] fp32 state before segment 0 (same on every rank), or None.
    Returns (out [T_r, H, dv], state after this rank's segment [H, dk, dv], state after the
    last segment [H, dk, dv]).
    """
    summary = summary or _default_summary
    scan = scan or _default_scan
    forward = forward or _default_forward
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    X, Z = summary(k, v, log_alpha, beta, l2norm)  # [1, H, dk, dk], [1, H, dk, dv]
    # gloo exchanges host tensors: the summaries cross over host memory and come back
    home = X.device
    via = torch.device("cpu") if dist.get_backend(group) == "gloo" else home
    X = X.to(via).contiguous()
    Z = Z.to(via).contiguous()
    xs = [torch.empty_like(X) for _ in range(world)]
    zs = [torch.empty_like(Z) for _ in range(world)]
    dist.all_gather(xs, X, group=group)
    dist.all_gather(zs, Z, group=group)
    E, S_last = scan(torch.cat(xs, 0).to(home), torch.cat(zs, 0).to(home), initial_state)
    out, S_mine = forward(q, k, v, log_alpha, beta, gate, E[rank], scale, l2norm)
    return out, S_mine, S_last
