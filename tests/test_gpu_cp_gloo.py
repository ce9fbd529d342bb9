"""Context parallelism over two ranks with the library's own kernels (needs a GPU).

K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context parallel": each
rank summarises its segment (kda_segment_summary), the fixed-size summaries are all-gathered,
every rank scans them in order (kda_scan_combine) and finishes its segment from the recovered
entry state (kda_chunk_fwd). Two gloo ranks run here as separate processes that both use
cuda:0; their kernels never wait on one another (the only exchange is the host-side
all-gather), so sharing one GPU is safe. The result is compared with the oracle's monolithic
recurrence over the whole sequence.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEG = [300, 213]  # tokens of rank 0 and rank 1 (ragged chunks)
H, D = 2, 128
SEED = 600


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from linear_attention_05_gb300 import cp, inputs
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    x = inputs.tokens(sum(SEG), H, D, D, torch.bfloat16, seed=SEED, device="cuda")
    S0 = inputs.state(1, H, D, D, seed=SEED + 1, device="cuda")[0].contiguous()
    lo = sum(SEG[:rank])
    t = {n: a[lo:lo + SEG[rank]].contiguous() for n, a in x.items()}
    out, s_mine, s_last = cp.context_parallel_forward(
        t["q"], t["k"], t["v"], t["log_alpha"], t["beta"], t["gate"], S0, scale=0.9)
    torch.cuda.synchronize()
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), out=out.float().cpu().numpy(),
             s_mine=s_mine.cpu().numpy(), s_last=s_last.cpu().numpy())
    dist.destroy_process_group()


def test_two_ranks_library_kernels_match_oracle(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    import oracle
    from linear_attention_05_gb300 import inputs
    from util import TOL, check
    # the same device generator as the ranks (CPU and CUDA generators draw different values)
    x = inputs.tokens(sum(SEG), H, D, D, torch.bfloat16, seed=SEED, device="cuda")
    f = {n: a.float().cpu().numpy() for n, a in x.items()}
    S0 = inputs.state(1, H, D, D, seed=SEED + 1, device="cuda").double().cpu().numpy()
    T = sum(SEG)
    ref_out, ref_S = oracle.forward(f["q"], f["k"], f["v"], f["log_alpha"], f["beta"], f["gate"],
                                    S0, [0, T], scale=0.9)
    _, ref_S0 = oracle.forward(f["q"], f["k"], f["v"], f["log_alpha"], f["beta"], f["gate"],
                               S0, [0, T], scale=0.9, t_stop=[SEG[0]])
    r0 = np.load(os.path.join(tmp_path, "rank0.npz"))
    r1 = np.load(os.path.join(tmp_path, "rank1.npz"))
    tol = TOL[torch.bfloat16]
    check("cp_two_ranks/out", np.concatenate([r0["out"], r1["out"]]), ref_out, tol)
    check("cp_two_ranks/state_after_rank0", r0["s_mine"], ref_S0[0], tol)
    check("cp_two_ranks/state_after_rank1", r1["s_mine"], ref_S[0], tol)
    for r in (r0, r1):
        check("cp_two_ranks/final_state", r["s_last"], ref_S[0], tol)
