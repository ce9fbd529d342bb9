"""Multi-rank host logic on CPU (gloo, world size 2), no GPU.

* Context parallelism (linear_attention_05_gb300.cp): each rank owns one segment of
  a sequence; the fixed-size segment summaries are all-gathered, scanned in order,
  and every rank finishes its segment from the recovered entry state. The compute
  steps are the fp64 oracle here, so the test checks the exchange itself: the
  ranks' outputs and states must equal one monolithic recurrence.
* bench.py's timing reduction across ranks (max over ranks).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SEG = [23, 41]          # tokens of rank 0 and rank 1 (ragged)
H, DK, DV = 2, 8, 6


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    r = np.random.default_rng(2024)
    T = sum(SEG)
    f = np.float32
    return {
        "q": r.standard_normal((T, H, DK)).astype(f),
        "k": r.standard_normal((T, H, DK)).astype(f),
        "v": r.standard_normal((T, H, DV)).astype(f),
        "log_alpha": np.maximum(-np.exp(r.standard_normal((T, H, DK)) - 2.0), np.log(0.5)).astype(f),
        "beta": (1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))).astype(f),
        "gate": (1.0 / (1.0 + np.exp(-r.standard_normal((T, H, DV))))).astype(f),
        "S0": 0.3 * r.standard_normal((H, DK, DV)),
    }


def _oracle_steps():
    import oracle

    def summary(k, v, la, b, l2norm):
        X, Z = oracle.segment_summary(k.numpy(), v.numpy(), la.numpy(), b.numpy(), [0, k.shape[0]],
                                      l2norm=l2norm)
        return torch.from_numpy(X), torch.from_numpy(Z)

    def scan(X, Z, S_init):
        E, Sf = oracle.scan_combine(X.numpy(), Z.numpy(), None if S_init is None else S_init.numpy())
        return torch.from_numpy(E), torch.from_numpy(Sf)

    def forward(q, k, v, la, b, g, entry, scale, l2norm):
        out, Sf = oracle.forward(q.numpy(), k.numpy(), v.numpy(), la.numpy(), b.numpy(),
                                 None if g is None else g.numpy(), entry.numpy()[None],
                                 [0, q.shape[0]], scale=scale, l2norm=l2norm)
        return torch.from_numpy(out), torch.from_numpy(Sf[0])

    return summary, scan, forward


def _cp_worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    from linear_attention_05_gb300 import cp
    x = _inputs()
    lo = sum(SEG[:rank])
    hi = lo + SEG[rank]
    t = {n: torch.from_numpy(np.ascontiguousarray(a[lo:hi])) for n, a in x.items() if n != "S0"}
    summary, scan, forward = _oracle_steps()
    out, s_mine, s_last = cp.context_parallel_forward(
        t["q"], t["k"], t["v"], t["log_alpha"], t["beta"], t["gate"],
        torch.from_numpy(x["S0"]), scale=0.9, summary=summary, scan=scan, forward=forward)
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), out=out.numpy(), s_mine=s_mine.numpy(),
             s_last=s_last.numpy())
    dist.destroy_process_group()


def _bench_worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    import bench
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 + rank, world)
    np.save(os.path.join(outdir, f"max{rank}.npy"), np.array([m]))
    dist.destroy_process_group()


def test_context_parallel_exchange_matches_monolithic(tmp_path):
    mp.spawn(_cp_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    import oracle
    x = _inputs()
    T = sum(SEG)
    ref_out, ref_S = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                                    x["S0"][None], [0, T], scale=0.9)
    _, ref_S0 = oracle.forward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                               x["S0"][None], [0, T], scale=0.9, t_stop=[SEG[0]])
    r0 = np.load(os.path.join(tmp_path, "rank0.npz"))
    r1 = np.load(os.path.join(tmp_path, "rank1.npz"))
    out = np.concatenate([r0["out"], r1["out"]])
    scale = np.max(np.abs(ref_out))
    assert np.max(np.abs(out - ref_out)) / scale < 1e-12
    assert np.max(np.abs(r0["s_mine"] - ref_S0[0])) < 1e-12
    assert np.max(np.abs(r1["s_mine"] - ref_S[0])) < 1e-12
    for r in (r0, r1):
        assert np.max(np.abs(r["s_last"] - ref_S[0])) < 1e-12


def test_bench_max_over_ranks(tmp_path):
    mp.spawn(_bench_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert float(np.load(os.path.join(tmp_path, f"max{r}.npy"))[0]) == 2.5


def test_bench_launches_its_own_ranks():
    """bench.py --gpus 2 outside torchrun starts the two ranks itself (the reference arm runs on
    the host cores, so this needs no GPU): rank 0 prints one JSON line with n_gpus 2, the other
    rank exits 0 without work."""
    import json
    import subprocess
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl",
                        "reference", "--steps", "1", "--warmup", "3", "--ref-tokens", "16"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_bench_rejects_gpus_that_differ_from_world_size():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl",
                        "reference", "--steps", "1"], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 2
    assert "WORLD_SIZE=1" in r.stderr
