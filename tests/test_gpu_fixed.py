"""Fixed-length batches on the tensor-core path (needs a GPU).

Without cu_seqlens the card and state kernels index the sequences in closed form and no chunk
table is launched. The same batch passed with cu_seqlens goes through the table; the two must
agree bit for bit (every chain is computed the same way), and both with the oracle (the plain
recurrence, K3 training overview section 2) on sampled chains. The lengths leave a ragged
last chunk, through the persistent prefill (few chains: one launch) and the two-kernel
schedule.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, np32, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.mark.parametrize("n_seq,L,H,launches", [
    (2, 1100, 4, 1),     # 18 chunks, the last of 12 tokens: the persistent prefill
    (8, 700, 16, 2),     # 128 (sequence, head) pairs: cards, then the state pass
    (3, 50, 2, 2),       # one partial chunk per sequence
])
def test_fixed_length_equals_varlen_and_oracle(n_seq, L, H, launches):
    T = n_seq * L
    assert B.kda_chunk_fwd_launches(T, n_seq, H, D, D) == launches
    x = inputs.tokens(T, H, D, D, torch.bfloat16, seed=91 + L, device=DEV)
    s0 = inputs.state(n_seq, H, D, D, seed=92 + L, device=DEV)
    outs = []
    for cu in (None, torch.arange(0, T + 1, L, dtype=torch.int32, device=DEV)):
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
        fs = torch.empty((n_seq, H, D, D), dtype=torch.float32, device=DEV)
        B.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, s0,
                        fs, cu, n_seq, scale=0.9)
        torch.cuda.synchronize()
        assert B.kda_get_error() == B.KDA_OK
        outs.append((out, fs))
    (o1, f1), (o2, f2) = outs
    assert torch.equal(o1, o2)
    assert torch.equal(f1, f2)
    for s, h in ((0, 0), (n_seq - 1, H - 1)):
        rows = slice(s * L, (s + 1) * L)
        g = lambda t: np32(t[rows, h:h + 1])
        ro, rs = oracle.forward(g(x["q"]), g(x["k"]), g(x["v"]), g(x["log_alpha"]),
                                np32(x["beta"][rows, h:h + 1]), g(x["gate"]),
                                np32(s0[s:s + 1, h:h + 1]).astype(np.float64), [0, L], scale=0.9)
        assert rel_err(np32(o1[rows, h:h + 1]), ro) <= TOL[torch.bfloat16]
        assert rel_err(np32(f1[s:s + 1, h:h + 1]), rs) <= TOL[torch.bfloat16]
