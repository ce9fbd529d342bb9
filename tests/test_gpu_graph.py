"""kda_chunk_fwd captured in a CUDA graph (needs a GPU).

A split prefill forks its trailing card launch onto a library stream and joins it back with
events, all ordered on the caller's stream; the persistent prefill clears its flags with a
memset on the caller's stream and makes one cooperative launch. Either call can be captured
and replayed.
A replay must give the eager call's bits, and, after the inputs are overwritten in place,
the new inputs' results.
"""
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, D, N_SEQ, L = 4, 128, 2, 1024   # 8 chains of 16 chunks: the split schedule


def _make(seed):
    x = inputs.tokens(N_SEQ * L, H, D, D, torch.bfloat16, seed=seed, device=DEV)
    s0 = inputs.state(N_SEQ, H, D, D, seed=seed + 1, device=DEV)
    return x, s0


@pytest.mark.parametrize("varlen", [True, False])
def test_split_prefill_graph_replay_is_bitwise_eager(varlen):
    """varlen: the split schedule (chunk table, then cards and state passes on two streams);
    fixed lengths: the persistent prefill (a flag reset and one cooperative launch)."""
    T = N_SEQ * L
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device=DEV) if varlen else None
    assert B.kda_chunk_fwd_launches(T, N_SEQ, H, D, D, varlen=varlen) == (5 if varlen else 1)
    x, s0 = _make(81)
    ws = torch.empty(B.kda_chunk_fwd_workspace_size(T, N_SEQ, H, D, D), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    fs = torch.empty((N_SEQ, H, D, D), dtype=torch.float32, device=DEV)

    def call():
        B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, s0, fs,
                        cu, N_SEQ, workspace=ws)

    call()
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    out_e, fs_e = out.clone(), fs.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    out.zero_()
    fs.zero_()
    with torch.cuda.graph(graph):
        call()
    graph.replay()
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    assert torch.equal(out, out_e)
    assert torch.equal(fs, fs_e)

    # new inputs written in place: the replay follows them
    x2, s02 = _make(83)
    for n in ("q", "k", "v", "log_alpha", "beta", "gate"):
        x[n].copy_(x2[n])
    s0.copy_(s02)
    graph.replay()
    torch.cuda.synchronize()
    out_g, fs_g = out.clone(), fs.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out)
    assert torch.equal(fs_g, fs)
    assert not torch.equal(out_g, out_e)
