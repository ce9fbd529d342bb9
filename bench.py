"""KDA benchmark: one JSON line on rank 0.

Workload (one "step"): chunked prefill of 4 sequences x 4096 tokens, 16 heads,
dk = dv = 128, bf16 inputs, fp32 initial state ~ N(0, 0.01) in, final state
out (one kda_chunk_fwd call). Inputs (~400 MB) are larger than the 129 MB L2,
so no flush is needed between steps. The JSON line also carries the decode
step (256 sequences x 32 heads, fp32 states in HBM) in GB/s of HBM traffic
and the long-context segment scan (1,048,576 tokens, 8 segments).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU (torchrun): every rank runs its own independent batch (weak
scaling, no collective on the data path); the timing is the max over ranks.
"--impl reference" times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = dict(B=4, T=4096, H=16, d=128)
TOKENS_PER_STEP = PREFILL["B"] * PREFILL["T"]
TOKEN_HEADS = TOKENS_PER_STEP * PREFILL["H"]
# algorithmic bytes of the prefill path per token-head (bf16 q, k, v, log_alpha,
# gate in; beta in; o out) and per (sequence, head) state (fp32 in + out)
BYTES_PER_TOKEN_HEAD = 5 * 128 * 2 + 2 + 128 * 2
STATE_BYTES = 128 * 128 * 4


PROFILE_OF = {"kda_card_tc": "kda_card_tc_prefill.md", "kda_state_tc": "kda_state_tc_prefill.md",
              "kda_prefill_fused": "kda_prefill_fused_persistent.md",
              "kda_decode_kernel": "kda_decode_kernel_decode.md",
              "kda_scan_tc": "kda_scan_tc_scan.md"}


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, or None when
    there is none or the kernel's source file changed since the counters were taken."""
    import hashlib
    import re
    name = PROFILE_OF.get(kernel)
    if name is None:
        return None
    try:
        txt = open(os.path.join(ROOT, "profiles", name)).read()
        mh = re.search(r"source_sha256: ([0-9a-f]+) \(([^)]+)\)", txt)
        mt = re.search(r"traffic_bytes_per_launch: (\d+)", txt)
        if not mh or not mt:
            return None
        h = hashlib.sha256()
        for f in mh.group(2).split(", "):  # the sources the kernel is built from, in order
            h.update(open(os.path.join(ROOT, f), "rb").read())
        cur = h.hexdigest()
        return int(mt.group(1)) if cur[:16] == mh.group(1) else None
    except OSError:
        return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """SM clock and clock-event reasons sampled in a background thread every 2 ms through
    NVML (libnvidia-ml, read-only queries), so that even a timed region of a few
    milliseconds holds several samples. Falls back to `nvidia-smi -lms 20` when NVML cannot
    be loaded."""

    # clock-event reason bits of NVML (nvmlClocksEventReason*)
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.device = device
        self.samples = []  # (monotonic time, sm MHz, max sm MHz, set of reason names)
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(self.device), "uuid", None)
        ok = False
        if uuid is not None:
            txt = str(uuid)
            txt = txt if txt.startswith("GPU-") else "GPU-" + txt
            ok = nv.nvmlDeviceGetHandleByUUID(txt.encode(), ctypes.byref(h)) == 0
        if not ok:
            idx = self.device.index or 0
            if "CUDA_VISIBLE_DEVICES" in os.environ:
                idx = int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[idx])
            if nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        return nv, h

    def start(self):
        try:
            import ctypes
            nv, h = self._nvml_handle()
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons

            def poll():
                clk, bits = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self.stop_flag.is_set():
                    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                            reasons_fn(h, ctypes.byref(bits)) == 0:
                        names = {n for b, n in self.REASONS.items() if bits.value & b}
                        self.samples.append((time.monotonic(), float(clk.value),
                                             float(mx.value), names))
                    time.sleep(0.002)

            self.thread = threading.Thread(target=poll, daemon=True)
            self.source = "nvml 2 ms"
            self.thread.start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.source = "nvidia-smi 20 ms"
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        for line in self.proc.stdout:
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 8 and num(p[0]) is not None:
                self.samples.append((time.monotonic(), num(p[0]), num(p[1]),
                                     {names[i] for i in range(4)
                                      if p[4 + i].lower().startswith("active")}))

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        note = []
        if not inside:  # window shorter than the sampling period: nearest sample
            inside = [min(self.samples, key=lambda x: abs(x[0] - 0.5 * (t0 + t1)))]
            note = ["window_shorter_than_sampling"]
        sm = [x[1] for x in inside if x[1] is not None]
        mx = [x[2] for x in inside if x[2] is not None]
        reasons = sorted(set().union(*[x[3] for x in inside]))
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons + note,
                "samples": len(inside), "source": self.source,
                "window_ms": round((t1 - t0) * 1e3, 2)}


def dist_setup(n_gpus):
    """Rank, world size and local rank from the torchrun environment (WORLD_SIZE must equal
    n_gpus; main() checks it or launches the ranks itself)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle
_CPU_INPUTS = {}


def oracle_prefill_sample(n_tokens: int, threads: int = 0):
    """Time the fp64 oracle on the first n_tokens of each of the 4 sequences
    of the prefill workload (all 16 heads). Returns (seconds, token count)."""
    import oracle
    from linear_attention_05_gb300 import inputs

    if "prefill" not in _CPU_INPUTS:
        _CPU_INPUTS["prefill"] = inputs.make("prefill", device="cpu")
    x = _CPU_INPUTS["prefill"]
    B_, T_ = PREFILL["B"], PREFILL["T"]
    idx = np.concatenate([np.arange(b * T_, b * T_ + n_tokens) for b in range(B_)])

    def sel(t):
        return t[idx].float().numpy()

    args = [sel(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "gate")]
    S0 = x["S0"].double().numpy()
    cu = [i * n_tokens for i in range(B_ + 1)]
    t0 = time.perf_counter()
    oracle.forward(*args, S0, cu, n_threads=threads)
    dt = time.perf_counter() - t0
    return dt, B_ * n_tokens, oracle.threads() if threads == 0 else threads


def cpu_baseline(target_s: float = 12.0):
    # calibrate on a small sample, then size the measured sample to ~target_s
    dt, ntok, cores = oracle_prefill_sample(64)
    per_tok = dt / ntok
    n = int(min(PREFILL["T"], max(64, target_s / per_tok / PREFILL["B"])))
    dt, ntok, cores = oracle_prefill_sample(n)
    # the same oracle on one thread, on a sample a sixteenth as long
    n1 = max(16, n // 16)
    dt1, ntok1, _ = oracle_prefill_sample(n1, threads=1)
    return {"value": ntok / dt / 1e6, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} tokens of each of the 4 sequences x 16 heads "
                      f"({ntok} tokens, {ntok * 16} token-heads) in {dt:.2f} s",
            "one_thread": {"value": ntok1 / dt1 / 1e6, "unit": "Mtok/s",
                           "sample": f"first {n1} tokens of each sequence in {dt1:.2f} s"}}


METRIC = "KDA prefill Mtok/s & % tensor peak; decode state GB/s vs GB300 HBM peak"


def prefill_config(world):
    return {"workload": "prefill B=4 T=4096 H=16 dk=dv=128 chunk=64, bf16 inputs, "
                        "fp32 initial/final state",
            "global_batch": PREFILL["B"] * world, "seq_len": PREFILL["T"],
            "parallelism": f"independent batch per GPU x{world}",
            "l2": "inputs (~400 MB) larger than L2; no flush"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    steps = []
    n_tok = None
    for i in range(args.warmup + args.steps):
        dt, ntok, cores = oracle_prefill_sample(args.ref_tokens)
        if i >= args.warmup:
            steps.append(dt)
            n_tok = ntok
    total = sum(steps)
    val = n_tok * len(steps) / total / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 6),
        "unit": "Mtok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(world),
        "cpu_baseline": {"value": round(val, 6), "unit": "Mtok/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"first {args.ref_tokens} tokens of each of the 4 sequences"
                                   f" x 16 heads per step"},
        "e2e": {"value": round(val, 6), "unit": "Mtok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def time_kernels(fn, steps, stream, n_launch):
    """Run fn() `steps` times with trace events around each of its launches;
    returns (total ms, per-launch-index list of ms)."""
    import linear_attention_05_gb300 as kda

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_launch)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for row in evs:  # create the events before the timed region
        for b, e in row:
            b.record(stream)
            e.record(stream)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        kda.kda_trace_events([b for b, _ in evs[i]], [e for _, e in evs[i]])
        fn()
    end.record(stream)
    kda.kda_trace_events([], [])
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    per = [sum(evs[i][j][0].elapsed_time(evs[i][j][1]) for i in range(steps)) / steps
           for j in range(n_launch)]
    return total, per


def run_gpu(args, rank, world, local):
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    kda.load()
    stream = torch.cuda.current_stream()

    w = inputs.WORKLOADS["prefill"]
    # every rank gets its own batch (weak scaling): shift the seed by rank
    w_rank = inputs.Workload(w.name, w.lengths, w.H, w.dk, w.dv, w.dtype, w.seed + 1000 * rank,
                             w.init_state)
    x = inputs.make(w_rank, device=dev)
    T, H, d = w.T_total, w.H, w.dk
    n_seq = len(w.lengths)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ws_bytes = kda.kda_chunk_fwd_workspace_size(T, n_seq, H, d, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                          x["S0"], fs, None, n_seq, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    # [chunk table,] cards, state pass; or for a split prefill [table,] leading cards, leading
    # state pass, trailing cards beside it, trailing state pass. The tensor-core path skips the
    # table for fixed-length batches (this workload passes no cu_seqlens).
    n_launch = kda.kda_chunk_fwd_launches(T, n_seq, H, d, d, varlen=False)
    total_ms, per_launch = time_kernels(step, args.steps, stream, n_launch)
    t_wall1 = time.monotonic()
    barrier(world)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * TOKENS_PER_STEP / (ms_per_step * 1e-3) / 1e6

    # roofline of the dominant kernel, over its launches per step: the persistent prefill (one
    # launch: cards and state pass together), or the update cards / state pass of the
    # two-kernel schedule
    tc = (w.dtype == torch.bfloat16 and d == 128)
    chunk_heads = (T // 64) * H
    fused = n_launch == 1
    if fused:
        names = ["kda_prefill_fused"]
        launches_of = [[0]]
        alg_bytes = {0: TOKEN_HEADS * BYTES_PER_TOKEN_HEAD + 2 * n_seq * H * STATE_BYTES}
        split = False
    else:
        names = (["kda_chunk_table", "kda_card_tc", "kda_state_tc"] if tc else
                 ["kda_chunk_table", "kda_prep_simt", "kda_state_simt"])
        has_table = n_launch in (3, 5)
        k0 = 1 if has_table else 0
        split = (n_launch - k0) == 4
        launches_of = [[0] if has_table else [],
                       [k0, k0 + 2] if split else [k0],
                       [k0 + 1, k0 + 3] if split else [k0 + 1]]
        alg_bytes = {  # algorithmic HBM bytes per step of each kernel
            0: (n_seq + 1) * 4 if has_table else 0,
            1: TOKEN_HEADS * (4 * d * 2 + 2),                                 # q, k, v, log_alpha, beta
            2: TOKEN_HEADS * (2 * d * 2) + 2 * n_seq * H * STATE_BYTES,       # gate, o, states
        }
    kernel_ms = [sum(per_launch[i] for i in ix) for ix in launches_of]  # per step
    dom = int(np.argmax(kernel_ms))
    n_dom = len(launches_of[dom])
    achieved = alg_bytes[dom] / (kernel_ms[dom] * 1e-3) / 1e9  # = per-launch bytes / mean duration
    traffic = profiled_traffic(names[dom])
    roofline = {"bound": "hbm", "kernel": names[dom], "achieved": round(achieved, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic, "peak_source": pk["source"],
                "launches_per_step": n_dom,
                "alg_bytes_per_launch": alg_bytes[dom] // n_dom,
                "launch_ms": {"per_step": dict(zip(names, [round(t, 4) for t in kernel_ms])),
                              "in_order": [round(t, 4) for t in per_launch]}}
    # the whole step against HBM: the path's algorithmic bytes over the step time
    step_bytes = sum(alg_bytes.values())
    roofline["step"] = {"alg_bytes": step_bytes,
                        "achieved": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                        "frac": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
    if split:
        roofline["schedule"] = ("split prefill: the cards of each sequence's trailing chunks are "
                                "built beside the state pass over its leading chunks")
    if fused:
        roofline["schedule"] = ("persistent prefill: one cooperative launch; all SMs build update "
                                "cards chunk-major, then one CTA per chain walks its chain while "
                                "the others build the remaining cards")
    if tc:
        # tensor-core work per (chunk, head): card GEMMs 1-4 and the state-pass MMA group,
        # over the whole step (the launches overlap, so their durations do not add up)
        card_flop = 2 * (128 * 64 * 128 + 2 * 128 * 64 * 64 + 2 * 128 * 64 * 64 + 2 * 128 * 128 * 64)
        state_flop = 2 * 128 * 192 * 128
        tf = chunk_heads * (card_flop + state_flop) / (ms_per_step * 1e-3) / 1e12
        roofline["tensor"] = {"kernels": names if fused else names[1:], "achieved": round(tf, 2), "unit": "TFLOP/s",
                              "peak": pk["bf16_tflops"], "frac": round(tf / pk["bf16_tflops"], 4),
                              "flop_per_chunk_head": card_flop + state_flop, "over": "step"}

    # end to end through the C ABI with host buffers: kda_chunk_fwd_host copies each sequence's
    # page-locked inputs in, computes it and copies its outputs back (copies on the library's
    # two copy streams, compute on this stream), so the transfers of one sequence overlap the
    # work on its neighbours; the last sequence is computed in four time slices, so that little
    # compute and copy-back is left after the last copy in.
    host = {k: v.to("cpu").pin_memory() for k, v in x.items() if k != "cu_seqlens" and v is not None}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size() + fs_h.numel() * fs_h.element_size()
    tail = 4
    dbuf = torch.empty(kda.kda_chunk_fwd_host_buffer_size(T, n_seq, H, d, d, tail_slices=tail),
                       dtype=torch.uint8, device=dev)

    def e2e_step():
        kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["log_alpha"], host["beta"],
                               host["gate"], out_h, host["S0"], fs_h, n_seq, tail_slices=tail,
                               device_buffer=dbuf, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    e2e = {"value": round(world * TOKENS_PER_STEP / (e2e_ms * 1e-3) / 1e6, 3), "unit": "Mtok/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms, 4), "api": "kda_chunk_fwd_host",
           "overlap": "per-sequence copy/compute pipeline, last sequence in 4 time slices"}
    del host, dbuf

    line = {
        "metric": METRIC,
        "value": round(value, 3), "unit": "Mtok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k unit-norm N(0,1), v N(0,1), beta/gate sigmoid(N(0,1)), "
                "log_alpha max(-exp(N(-3,1)), log 0.5))",
        "config": prefill_config(world),
        "roofline": roofline, "e2e": e2e, "clocks": clocks,
        "gpu_launches": n_launch * args.steps,
    }

    if rank == 0 and not args.skip_extra:
        line["decode"] = bench_decode(dev, pk, stream)
        line["varlen"] = bench_varlen(dev, pk, stream)
        line["segment_scan"] = bench_segment_scan(dev, pk, stream)
        line["scan_combine"] = bench_scan(dev, pk, stream)
        line["prefill_checkpoints"] = bench_checkpoints(dev, pk, stream)
        line["persistent_prefill"] = bench_persistent(dev, pk, stream)
        line["backward"] = bench_backward(dev, pk, stream)
        line["gate_prep"] = bench_gates(dev, pk, stream)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_decode(dev, pk, stream, steps=64):
    """256 sequences x 32 heads, fp32 state (512 MiB) resident; 64 steps, one
    kda_decode_step call per step with fresh inputs."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["decode"]
    N, H, d = len(w.lengths), w.H, w.dk
    S = inputs.state(N, H, d, d, w.seed, device=dev).contiguous()
    xs = [inputs.tokens(N, H, d, d, w.dtype, w.seed, step=s, device=dev) for s in range(steps)]
    outs = [torch.empty((N, H, d), dtype=w.dtype, device=dev) for _ in range(steps)]

    def run(i):
        x = xs[i]
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"],
                            outs[i], S, stream=stream)

    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for b, e in evs:
        b.record(stream)
        e.record(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        kda.kda_trace_events([evs[i][0]], [evs[i][1]])
        run(i)
    t1.record(stream)
    kda.kda_trace_events([], [])
    torch.cuda.synchronize()
    per_step_ms = t0.elapsed_time(t1) / steps
    kern_ms = sum(b.elapsed_time(e) for b, e in evs) / steps
    bytes_step = 2 * N * H * STATE_BYTES + N * H * (5 * d * 2 + 2 + d * 2)
    gbs = bytes_step / (kern_ms * 1e-3) / 1e9
    return {"workload": "decode 256 seq x 32 heads, dk=dv=128, bf16 tokens, fp32 state, 64 steps",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_step": round(per_step_ms * 1e3, 2),
            "kernel_us": round(kern_ms * 1e3, 2),
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": round(gbs, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": profiled_traffic("kda_decode_kernel"),
                         "bytes_per_launch": bytes_step},
            "gpu_launches": steps}


def bench_segment_scan(dev, pk, stream, reps=2):
    """1,048,576 tokens x 16 heads, 8 segments of 131,072: summaries, ordered
    scan, segment re-run from the recovered entry states."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["longctx"]
    T, H, d, n_seg = w.T_total, w.H, w.dk, w.n_segments
    x = inputs.make(w, device=dev)
    cu = torch.arange(0, T + 1, T // n_seg, dtype=torch.int32, device=dev)
    X = torch.empty((n_seg, H, d, d), dtype=torch.float32, device=dev)
    Z = torch.empty((n_seg, H, d, d), dtype=torch.float32, device=dev)
    E = torch.empty_like(Z)
    Sf = torch.empty((H, d, d), dtype=torch.float32, device=dev)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seg, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(T, n_seg, H, d, d), dtype=torch.uint8,
                     device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def run(record):
        if record:
            ev[0].record(stream)
        kda.kda_segment_summary(x["k"], x["v"], x["log_alpha"], x["beta"], cu, n_seg, X, Z,
                                workspace=ws, stream=stream)
        if record:
            ev[1].record(stream)
        kda.kda_scan_combine(X, Z, None, E, Sf, stream=stream)
        if record:
            ev[2].record(stream)
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out, E,
                          fs, cu, n_seg, workspace=ws, stream=stream)
        if record:
            ev[3].record(stream)

    run(False)
    torch.cuda.synchronize()
    tot = [0.0, 0.0, 0.0]
    for _ in range(reps):
        run(True)
        torch.cuda.synchronize()
        for i in range(3):
            tot[i] += ev[i].elapsed_time(ev[i + 1]) / reps
    th = T * H
    scan_bytes = n_seg * H * (d * d + d * d) * 4 + n_seg * H * d * d * 4 + H * d * d * 4
    # the same scheme in one call that computes the update cards once (kda_segmented_fwd)
    del ws
    wsf = torch.empty(kda.kda_segmented_fwd_workspace_size(T, n_seg, H, d, d), dtype=torch.uint8,
                      device=dev)
    fsf = torch.empty((H, d, d), dtype=torch.float32, device=dev)

    def fused():
        kda.kda_segmented_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                              None, fsf, None, cu, n_seg, workspace=wsf, stream=stream)

    fused()
    torch.cuda.synchronize()
    ev[0].record(stream)
    for _ in range(reps):
        fused()
    ev[1].record(stream)
    torch.cuda.synchronize()
    fused_ms = ev[0].elapsed_time(ev[1]) / reps
    return {"workload": "long context T=1,048,576 H=16 dk=dv=128 bf16, 8 segments",
            "summary_ms": round(tot[0], 3), "scan_ms": round(tot[1], 4),
            "rerun_ms": round(tot[2], 3),
            "three_calls_value": round(T / ((tot[0] + tot[1] + tot[2]) * 1e-3) / 1e6, 3),
            "fused_ms": round(fused_ms, 3),
            "value": round(T / (fused_ms * 1e-3) / 1e6, 3), "unit": "Mtok/s",
            "scan_gbs": round(scan_bytes / (tot[1] * 1e-3) / 1e9, 1),
            "summary_alg_gbs": round(th * (3 * d * 2 + 2) / (tot[0] * 1e-3) / 1e9, 1),
            "gpu_launches": 12 * reps}


def bench_varlen(dev, pk, stream, reps=10):
    """8 packed sequences (lengths drawn from [1024, 32768], about 112K tokens), 32 heads,
    dk=dv=128, bf16, zero initial state: kda_chunk_fwd with cu_seqlens."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["varlen"]
    x = inputs.make(w, device=dev)
    T, H, d, n_seq = w.T_total, w.H, w.dk, len(w.lengths)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(T, n_seq, H, d, d), dtype=torch.uint8,
                     device=dev)

    def run():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                          None, fs, x["cu_seqlens"], n_seq, workspace=ws, stream=stream)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    return {"workload": f"varlen {n_seq} packed sequences ({T} tokens, longest "
                        f"{max(w.lengths)}) H=32 dk=dv=128 bf16",
            "value": round(T / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s", "ms": round(ms, 3),
            "gpu_launches": kda.kda_chunk_fwd_launches(T, n_seq, H, d, d, varlen=True) * reps}


def bench_checkpoints(dev, pk, stream, reps=20, every=1024):
    """The prefill workload with prefix-cache checkpoints every 1024 tokens
    (kda_chunk_fwd_checkpoints), timed beside the same call without them."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=dev)
    T, H, d, n_seq = w.T_total, w.H, w.dk, len(w.lengths)
    per = w.lengths[0] // every
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ck = torch.empty((n_seq, per, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(T, n_seq, H, d, d), dtype=torch.uint8,
                     device=dev)

    def plain():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                          x["S0"], fs, None, n_seq, workspace=ws, stream=stream)

    def with_ckpt():
        kda.kda_chunk_fwd_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                      x["gate"], out, x["S0"], fs, ck, every, None, n_seq,
                                      workspace=ws, stream=stream)

    ms = {}
    for name, fn in (("plain", plain), ("ckpt", with_ckpt)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / reps
    return {"workload": "prefill B=4 T=4096 H=16 dk=dv=128 bf16, a checkpoint every 1024 "
                        "tokens (4 per sequence)",
            "value": round(T / (ms["ckpt"] * 1e-3) / 1e6, 3), "unit": "Mtok/s",
            "ms": round(ms["ckpt"], 4), "ms_without": round(ms["plain"], 4),
            "checkpoint_bytes": ck.numel() * 4,
            "gpu_launches": kda.kda_chunk_fwd_launches(T, n_seq, H, 128, 128, varlen=False) * reps}


def bench_backward(dev, pk, stream, reps=5):
    """kda_chunk_bwd on the prefill workload (bf16 inputs, fp32 arithmetic): gradients of
    <d_out, o> + <d_final, S_final> for all seven inputs."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=dev)
    T, H, d, n_seq = w.T_total, w.H, w.dk, len(w.lengths)
    g = torch.Generator(device=dev).manual_seed(99)
    d_out = torch.randn((T, H, d), generator=g, device=dev).to(torch.bfloat16)
    d_fin = torch.randn((n_seq, H, d, d), generator=g, device=dev)
    grads = {n: torch.empty_like(x[n]) for n in ("q", "k", "v", "log_alpha", "beta", "gate")}
    dS0 = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_bwd_workspace_size(T, n_seq, H, d, d), dtype=torch.uint8,
                     device=dev)

    def step():
        kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], x["S0"],
                          d_out, d_fin, grads["q"], grads["k"], grads["v"], grads["log_alpha"],
                          grads["beta"], grads["gate"], dS0, None, n_seq, workspace=ws,
                          stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    return {"workload": "backward of prefill B=4 T=4096 H=16 dk=dv=128, bf16 in/out, fp32 "
                        "arithmetic (batched contractions and both state passes on the tensor cores)",
            "value": round(T / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s", "ms": round(ms, 3),
            "workspace_bytes": ws.numel(), "gpu_launches": 15 * reps}


def bench_gates(dev, pk, stream, reps=20):
    """The prefill workload taking gate logits: kda_chunk_fwd with KDA_GATE_LOGITS (the
    sigmoids and the log-retention bound applied as the kernels load their inputs),
    timed beside an element-wise pre-pass (torch) followed by the plain call."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    w = inputs.WORKLOADS["prefill"]
    x = inputs.make(w, device=dev)
    T, H, d, n_seq = w.T_total, w.H, w.dk, len(w.lengths)
    g = torch.Generator(device=dev).manual_seed(5)
    raw = {"a": (torch.randn((T, H, d), generator=g, device=dev) - 3.0).to(torch.bfloat16),
           "bx": torch.randn((T, H), generator=g, device=dev).to(torch.bfloat16),
           "gx": torch.randn((T, H, d), generator=g, device=dev).to(torch.bfloat16)}
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(T, n_seq, H, d, d), dtype=torch.uint8,
                     device=dev)
    half = float(np.log(0.5))

    def fused():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], raw["a"], raw["bx"], raw["gx"], out, x["S0"],
                          fs, None, n_seq, flags=kda.KDA_QK_L2NORM | kda.KDA_GATE_LOGITS,
                          workspace=ws, stream=stream)

    def unfused():
        la = torch.clamp_min(-torch.exp(raw["a"].float()), half).to(torch.bfloat16)
        b = torch.sigmoid(raw["bx"].float()).to(torch.bfloat16)
        gt = torch.sigmoid(raw["gx"].float()).to(torch.bfloat16)
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], la, b, gt, out, x["S0"], fs, None, n_seq,
                          workspace=ws, stream=stream)

    ms = {}
    for name, fn in (("fused", fused), ("unfused", unfused)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / reps
    return {"workload": "prefill B=4 T=4096 H=16 dk=dv=128 bf16 with beta/gate logits and the "
                        "forget-gate pre-activation",
            "value": round(T / (ms["fused"] * 1e-3) / 1e6, 3), "unit": "Mtok/s",
            "ms": round(ms["fused"], 4), "ms_prepass_then_plain": round(ms["unfused"], 4),
            "gpu_launches": kda.kda_chunk_fwd_launches(T, n_seq, H, 128, 128, varlen=False) * reps}


def bench_persistent(dev, pk, stream, reps=20):
    """Fixed-length prefill with few chains (2 x 8192 tokens, 16 heads: 32 chains of 128
    chunks), where kda_chunk_fwd takes the persistent prefill (one cooperative launch), timed
    beside the same problem through the two-kernel schedule (the lengths passed as cu_seqlens)."""
    import linear_attention_05_gb300 as kda
    from linear_attention_05_gb300 import inputs

    n_seq, L, H, d = 2, 8192, 16, 128
    T = n_seq * L
    x = inputs.tokens(T, H, d, d, torch.bfloat16, seed=11, device=dev)
    S0 = inputs.state(n_seq, H, d, d, seed=12, device=dev)
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(T, n_seq, H, d, d), dtype=torch.uint8,
                     device=dev)
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device=dev)
    ms = {}
    for name, c in (("persistent", None), ("two_kernel", cu)):
        def fn():
            kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["gate"], out,
                              S0, fs, c, n_seq, workspace=ws, stream=stream)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / reps
    alg = T * H * BYTES_PER_TOKEN_HEAD + 2 * n_seq * H * STATE_BYTES
    return {"workload": "prefill 2 x 8192 tokens, H=16 (32 chains), dk=dv=128 bf16",
            "value": round(T / (ms["persistent"] * 1e-3) / 1e6, 3), "unit": "Mtok/s",
            "ms": round(ms["persistent"], 4), "ms_two_kernel": round(ms["two_kernel"], 4),
            "roofline": {"bound": "hbm", "kernel": "kda_prefill_fused",
                         "achieved": round(alg / (ms["persistent"] * 1e-3) / 1e9, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(alg / (ms["persistent"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                         "traffic": profiled_traffic("kda_prefill_fused")},
            "gpu_launches": reps * (kda.kda_chunk_fwd_launches(T, n_seq, H, d, d) +
                                    kda.kda_chunk_fwd_launches(T, n_seq, H, d, d, varlen=True))}


def bench_scan(dev, pk, stream, reps=20):
    """kda_scan_combine alone on long-context-sized summaries (8 segments x 16 heads). The
    inputs (26 MB) fit in L2, so L2 is flushed (a 256 MB write) before every call and each call
    is timed alone: the number is a cold-DRAM one."""
    import linear_attention_05_gb300 as kda

    n_seg, H, d = 8, 16, 128
    g = torch.Generator(device=dev).manual_seed(77)
    X = (torch.randn((n_seg, H, d, d), generator=g, device=dev) / d ** 0.5).contiguous()
    Z = torch.randn((n_seg, H, d, d), generator=g, device=dev).contiguous()
    E = torch.empty_like(Z)
    Sf = torch.empty((H, d, d), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        kda.kda_scan_combine(X, Z, None, E, Sf, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.fill_(1)
            e0.record(stream)
            kda.kda_scan_combine(X, Z, None, E, Sf, stream=stream)
            e1.record(stream)
    torch.cuda.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / reps
    kernel = "kda_scan_tc" if d == 128 else "kda_scan_kernel"
    nbytes = (2 * n_seg + n_seg + 1) * H * d * d * 4
    return {"workload": "scan combine, 8 segments x 16 heads, dk=dv=128, fp32", "kernel": kernel,
            "ms": round(ms, 4), "value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "frac": round(nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "l2": "flushed before every call", "traffic": profiled_traffic(kernel),
            "gpu_launches": reps}


def run_part(args, local):
    """One part of the path on its own (used for profiling a single kernel)."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    stream = torch.cuda.current_stream()
    fn = {"decode": bench_decode, "segscan": bench_segment_scan, "scan": bench_scan,
          "ckpt": bench_checkpoints, "bwd": bench_backward, "gates": bench_gates,
          "varlen": bench_varlen, "persistent": bench_persistent}[args.only]
    print(json.dumps({"part": args.only, **fn(dev, pk, stream)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=256,
                    help="reference arm: tokens per sequence timed per step")
    ap.add_argument("--skip-extra", action="store_true", help="prefill line only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", default=None, choices=["decode", "segscan", "scan", "ckpt", "bwd", "gates", "varlen",
                                                     "persistent"],
                    help="run one part of the path alone and print its numbers (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # launch the N ranks ourselves (one process per GPU, the same torchrun command a
        # multi-GPU driver uses) and pass their exit status on
        if args.impl != "reference" and torch.cuda.device_count() < args.gpus:
            print(f"bench.py: --gpus {args.gpus} but {torch.cuda.device_count()} visible GPUs",
                  file=sys.stderr)
            sys.exit(2)
        import socket
        with socket.socket() as sck:
            sck.bind(("127.0.0.1", 0))
            port = sck.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if world_env != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}", file=sys.stderr)
        sys.exit(2)
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.only:
        if rank == 0:
            run_part(args, local)
    else:
        run_gpu(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
