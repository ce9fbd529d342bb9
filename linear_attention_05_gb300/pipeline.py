"""kda_chunk_fwd on host-resident inputs, with the transfers overlapped.

For a batch of equal-length sequences held in pinned host memory, ``HostPipeline.run``
moves the batch in groups of sequences over three CUDA streams: the inputs of group
i + 1 are copied in while group i is computed and group i - 1 is copied out. Every
step of the computation is the library's kda_chunk_fwd on the group's sequences
(they are independent, so the results are bitwise those of one call on the whole
batch); this module only orders copies and calls.

With ``parts`` > 1 (one sequence per group), each sequence is also cut in time into
``parts`` slices of a multiple of 64 tokens; slice p starts from the state slice p - 1
left, so the results are still bitwise those of one call (the chunks are the same and the
fp32 state hand-over is exact), and the pipeline's tail after the last copy in is one
slice's compute and copy out instead of a whole sequence's. ``tail_parts`` cuts only the last
group that way: the tail shrinks while the other groups keep one call each (every call costs
host time to issue).
"""
from __future__ import annotations

import torch

from . import binding

_TOKEN = ("q", "k", "v", "log_alpha", "beta", "gate")


class HostPipeline:
    """Device buffers, workspace and streams for batches of ``n_seq`` sequences of
    ``seq_len`` tokens (``H`` heads, ``dk``/``dv``), processed in ``groups`` groups, each
    sequence in ``parts`` time slices (``parts`` > 1 needs one sequence per group)."""

    def __init__(self, n_seq, seq_len, H, dk, dv, dtype=torch.bfloat16, device="cuda",
                 groups=None, with_gate=True, parts=1, tail_parts=None):
        self.n_seq, self.L, self.H, self.dk, self.dv = n_seq, seq_len, H, dk, dv
        self.groups = groups or n_seq
        if n_seq % self.groups:
            raise ValueError("n_seq must be a multiple of groups")
        self.spg = n_seq // self.groups  # sequences per group
        self.parts = parts
        self.tail_parts = tail_parts or parts
        for pp in (parts, self.tail_parts):
            if pp > 1 and (self.spg != 1 or seq_len % pp or (seq_len // pp) % binding.CHUNK):
                raise ValueError("parts > 1 needs one sequence per group and slices of a multiple "
                                 "of 64 tokens")
        T = n_seq * seq_len
        dev = torch.device(device)
        shapes = {"q": (T, H, dk), "k": (T, H, dk), "v": (T, H, dv), "log_alpha": (T, H, dk),
                  "beta": (T, H), "gate": (T, H, dv)}
        self.dev_in = {n: torch.empty(s, dtype=dtype, device=dev) for n, s in shapes.items()
                       if with_gate or n != "gate"}
        self.dev_s0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
        self.dev_out = torch.empty((T, H, dv), dtype=dtype, device=dev)
        self.dev_fs = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
        # states handed between time slices, used alternately
        self.dev_mid = ([torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
                         for _ in range(2)] if max(parts, self.tail_parts) > 1 else [])
        tg = self.spg * seq_len // min(parts, self.tail_parts)  # tokens of the largest call
        nbytes = binding.kda_chunk_fwd_workspace_size(
            tg, self.spg, H, dk, dv, dtype=binding._dtype_code(self.dev_out))
        self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(dev), torch.cuda.Stream(dev),
                                              torch.cuda.Stream(dev))

    def run(self, host, out_host, final_state_host=None, scale=1.0, flags=binding.KDA_QK_L2NORM):
        """host: dict of pinned tensors q, k, v, log_alpha, beta, gate (optional) and S0
        (optional, [n_seq, H, dk, dv] fp32). Writes out_host (pinned [T, H, dv]) and, if given,
        final_state_host. Work is ordered after the current stream; the current stream waits
        for the last copy out."""
        cur = torch.cuda.current_stream()
        self.s_in.wait_stream(cur)
        self.s_comp.wait_stream(cur)
        self.s_out.wait_stream(cur)
        has_gate = host.get("gate") is not None
        has_s0 = host.get("S0") is not None
        for g in range(self.groups):
            s0, s1 = g * self.spg, (g + 1) * self.spg
            if has_s0:
                with torch.cuda.stream(self.s_in):
                    self.dev_s0[s0:s1].copy_(host["S0"][s0:s1], non_blocking=True)
            parts = self.tail_parts if g == self.groups - 1 else self.parts
            tp = self.spg * self.L // parts  # tokens of one call
            for p in range(parts):
                t0 = g * self.spg * self.L + p * tp
                t1 = t0 + tp
                with torch.cuda.stream(self.s_in):
                    for n in _TOKEN:
                        if n == "gate" and not has_gate:
                            continue
                        self.dev_in[n][t0:t1].copy_(host[n][t0:t1], non_blocking=True)
                self.s_comp.wait_stream(self.s_in)
                if p == 0:
                    entry = self.dev_s0[s0:s1] if has_s0 else None
                else:
                    entry = self.dev_mid[(p - 1) % 2][s0:s1]
                last = p == parts - 1
                exit_ = self.dev_fs[s0:s1] if last else self.dev_mid[p % 2][s0:s1]
                binding.kda_chunk_fwd(
                    self.dev_in["q"][t0:t1], self.dev_in["k"][t0:t1], self.dev_in["v"][t0:t1],
                    self.dev_in["log_alpha"][t0:t1], self.dev_in["beta"][t0:t1],
                    self.dev_in["gate"][t0:t1] if has_gate else None, self.dev_out[t0:t1],
                    entry, exit_, None, self.spg, scale=scale, flags=flags, workspace=self.ws,
                    stream=self.s_comp)
                self.s_out.wait_stream(self.s_comp)
                with torch.cuda.stream(self.s_out):
                    out_host[t0:t1].copy_(self.dev_out[t0:t1], non_blocking=True)
                    if last and final_state_host is not None:
                        final_state_host[s0:s1].copy_(self.dev_fs[s0:s1], non_blocking=True)
        cur.wait_stream(self.s_out)
        return out_host, final_state_host
