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


def test_backward_graph_replay_is_bitwise_eager():
    """kda_chunk_bwd forks the library's second stream off the caller's and joins it back (the
    two state passes run side by side); captured in a CUDA graph, the call replays bit for bit
    like the eager call and follows new inputs written in place."""
    lengths = [300, 129]
    T, n, Hb, d = sum(lengths), len(lengths), 2, 128
    x = inputs.tokens(T, Hb, d, d, torch.bfloat16, seed=85, device=DEV)
    s0 = inputs.state(n, Hb, d, d, seed=86, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(87)
    d_out = torch.randn((T, Hb, d), generator=g).to(torch.bfloat16).to(DEV)
    d_fin = torch.randn((n, Hb, d, d), generator=g).to(DEV)
    cu = torch.tensor([0, lengths[0], T], dtype=torch.int32, device=DEV)
    ws = torch.empty(B.kda_chunk_bwd_workspace_size(T, n, Hb, d, d), dtype=torch.uint8,
                     device=DEV)
    grads = {nm: torch.empty_like(x[src]) for nm, src in (
        ("dq", "q"), ("dk", "k"), ("dv", "v"), ("dlog_alpha", "log_alpha"), ("dbeta", "beta"),
        ("dgate", "gate"))}
    grads["dS0"] = torch.empty((n, Hb, d, d), dtype=torch.float32, device=DEV)

    def call():
        B.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], s0, d_out,
                        d_fin, grads["dq"], grads["dk"], grads["dv"], grads["dlog_alpha"],
                        grads["dbeta"], grads["dgate"], grads["dS0"], cu, n, workspace=ws)

    call()
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    eager = {nm: t.clone() for nm, t in grads.items()}

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    for t in grads.values():
        t.zero_()
    with torch.cuda.graph(graph):
        call()
    graph.replay()
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    for nm, t in grads.items():
        assert torch.equal(t, eager[nm]), nm

    # new inputs and cotangents written in place: the replay follows them
    x2 = inputs.tokens(T, Hb, d, d, torch.bfloat16, seed=89, device=DEV)
    for nm in ("q", "k", "v", "log_alpha", "beta", "gate"):
        x[nm].copy_(x2[nm])
    d_out.copy_(torch.randn((T, Hb, d), generator=g).to(torch.bfloat16).to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    replayed = {nm: t.clone() for nm, t in grads.items()}
    call()
    torch.cuda.synchronize()
    assert B.kda_get_error() == B.KDA_OK
    for nm, t in grads.items():
        assert torch.equal(replayed[nm], t), nm
    assert not torch.equal(replayed["dq"], eager["dq"])
