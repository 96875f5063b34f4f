"""Benchmark of the KDA hot path on one GB300 (or N independent replicas).

One step = one pass of the whole path over one batch of synthetic input:
  prefill : B=1, T=8192, H=12, d=128, initial state ~ N(0, 0.02^2), o in bf16
  decode  : 256 sequences x 96 heads, one token each, on a 1.6 GB fp32 state updated in place
value = (prefill + decode) token-heads per second over the whole job; the prefill and
decode parts are also reported on their own, with their roofline fractions.

Run:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 is launched with torchrun, one rank per GPU, each rank a full replica
(independent sequences, no collective on the data path: weak scaling).
--impl reference times the fp64 CPU oracle on this host's cores (a bounded sample of
the same workload per step).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_serving_02_gb300 import inputs  # noqa: E402

PREFILL_T, PREFILL_H = 8192, 12
DECODE_N, DECODE_H = 256, 96
D = 128
# algorithmic bytes per token-head
PREFILL_BYTES_PER_TH = 4 * 2 * D + 4 * D + 4          # q, k, v, o (bf16) + z (fp32) + b = 1540
DECODE_BYTES_PER_TH = 2 * 4 * D * D + 3 * 2 * D + 4 * D + 4 + 4 * D   # S read+write, q,k,v, z, b, o = 132868
# algorithmic tensor-core flops per token-head of the chunk form (C=64, triangles counted once)
PREFILL_FLOPS_PER_TH = 5 * 64 * D + 6 * D * D          # 139264
METRIC = "KDA prefill tokens/s·head & decode tokens/s at d=128 on 1 GB300; % of roofline"
WORKLOAD = ("prefill B=1 T=8192 H=12 d=128 (S0~N(0,0.02^2), o bf16) + decode N=256 H=96 d=128 "
            "(1 token/seq, 1.6 GB fp32 state in place)")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 10 ms while running (the
    timed region of a short run lasts tens of milliseconds)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------
# ranks
# ------------------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    """The largest x over all ranks (on the device with NCCL, on the host with gloo)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------
# workload
# ------------------------------------------------------------------------------------
DECODE_POOL = 16  # distinct decode-token batches, cycled through the steps


def make_workload(rank):
    """Prefill inputs (drawn on the host from the seeded generator, so the oracle sees the
    same tensors), the device-resident decode state, and a pool of decode-token batches
    that the steps cycle through (the state changes every step either way)."""
    seed = 1000 * rank
    pre_cpu = inputs.prefill_inputs(PREFILL_T, PREFILL_H, 1, seed=seed, init_state=True)
    pre = {k: v.cuda() for k, v in pre_cpu.items()}
    state = inputs.decode_state(DECODE_N, DECODE_H, seed=seed + 1, device="cuda")
    dec = [inputs.decode_step_inputs(DECODE_N, DECODE_H, seed=seed + 1, step=i, device="cuda")
           for i in range(DECODE_POOL)]
    return pre_cpu, pre, state, dec


class Flusher:
    """Writes a buffer larger than L2 (129 MB) between timed steps."""

    def __init__(self, nbytes=512 << 20):
        self.buf = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.buf.fill_(1.0)


def run_ours_device(pre, state, dec, steps, warmup, world):
    from linear_attention_serving_02_gb300 import kda

    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(PREFILL_T, 1, PREFILL_H), dtype=torch.uint8, device="cuda")
    o = torch.empty(pre["q"].shape, dtype=torch.bfloat16, device="cuda")
    S = torch.empty((1, PREFILL_H, D, D), dtype=torch.float32, device="cuda")
    o_dec = torch.empty((DECODE_N, DECODE_H, D), dtype=torch.float32, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def step(i):
        kda.kda_chunk_prefill(pre["q"], pre["k"], pre["v"], pre["z"], pre["A"], pre["b"], initial_state=pre["S0"],
                              o=o, final_state=S, workspace=ws)
        d = dec[i % len(dec)]
        kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["z"], d["A"], d["b"], state, o=o_dec)

    for i in range(warmup):
        flush()
        step(i)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        e0, e1, e2 = ev[j]
        d = dec[(warmup + j) % len(dec)]
        e0.record(stream)
        kda.kda_chunk_prefill(pre["q"], pre["k"], pre["v"], pre["z"], pre["A"], pre["b"], initial_state=pre["S0"],
                              o=o, final_state=S, workspace=ws)
        e1.record(stream)
        kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["z"], d["A"], d["b"], state, o=o_dec)
        e2.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    pre_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    finite = bool(torch.isfinite(S).all() and torch.isfinite(o_dec).all())
    return pre_ms, dec_ms, finite


def run_ours_e2e(pre_cpu, dec, steps, warmup, world):
    """Same step through the public API with host buffers: every step copies its inputs
    from pinned host memory to the device and its outputs back, inside the timed region,
    and the host waits for each step's outputs. The decode state stays resident on the
    device (it is the serving-side cache).

    Pipelined as a serving loop would be: inputs and outputs are double-buffered, step
    i + 1's inputs are uploaded on one copy stream while step i computes, step i's prefill
    outputs are read back on another while its decode runs, and the host takes step i's
    results while step i + 1 computes. Each step's working
    set (151 MB of prefill inputs, the 1.6 GB state) is larger than L2, so no flush runs
    between steps. Returns the total time of the timed steps."""
    from linear_attention_serving_02_gb300 import kda

    h_pre = {k: v.pin_memory() for k, v in pre_cpu.items()}
    h_dec = [{k: v.cpu().pin_memory() for k, v in d.items()} for d in dec]
    d_pre = [{k: torch.empty_like(v, device="cuda") for k, v in h_pre.items()} for _ in range(2)]
    d_dec = [{k: torch.empty_like(v, device="cuda") for k, v in h_dec[0].items()} for _ in range(2)]
    state = inputs.decode_state(DECODE_N, DECODE_H, seed=7, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(PREFILL_T, 1, PREFILL_H), dtype=torch.uint8, device="cuda")
    o = [torch.empty(h_pre["q"].shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    S = [torch.empty((1, PREFILL_H, D, D), dtype=torch.float32, device="cuda") for _ in range(2)]
    o_dec = [torch.empty((DECODE_N, DECODE_H, D), dtype=torch.float32, device="cuda") for _ in range(2)]
    h_o = [torch.empty(o[0].shape, dtype=o[0].dtype).pin_memory() for _ in range(2)]
    h_S = [torch.empty(S[0].shape, dtype=S[0].dtype).pin_memory() for _ in range(2)]
    h_od = [torch.empty(o_dec[0].shape, dtype=o_dec[0].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_pre.values()) + \
        sum(t.numel() * t.element_size() for t in h_dec[0].values())
    d2h = sum(t.numel() * t.element_size() for t in (h_o[0], h_S[0], h_od[0]))
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, pre_done, dec_done, out_ready = ([ev(), ev()] for _ in range(4))
    for b in range(2):  # nothing in flight yet: the first waits return at once
        dec_done[b].record(main)
        out_ready[b].record(down)

    def upload(i):
        b = i % 2
        with torch.cuda.stream(up):
            up.wait_event(dec_done[b])  # step i - 2 is done reading these buffers
            for k in d_pre[b]:
                d_pre[b][k].copy_(h_pre[k], non_blocking=True)
            for k in d_dec[b]:
                d_dec[b][k].copy_(h_dec[i % len(h_dec)][k], non_blocking=True)
            in_ready[b].record(up)

    def compute_and_read_back(i):
        b = i % 2
        main.wait_event(in_ready[b])
        main.wait_event(out_ready[b])  # step i - 2's outputs have left these buffers
        p = d_pre[b]
        kda.kda_chunk_prefill(p["q"], p["k"], p["v"], p["z"], p["A"], p["b"], initial_state=p["S0"], o=o[b],
                              final_state=S[b], workspace=ws)
        pre_done[b].record(main)
        q = d_dec[b]
        kda.kda_recurrent_decode(q["q"], q["k"], q["v"], q["z"], q["A"], q["b"], state, o=o_dec[b])
        dec_done[b].record(main)
        with torch.cuda.stream(down):
            down.wait_event(pre_done[b])
            h_o[b].copy_(o[b], non_blocking=True)
            h_S[b].copy_(S[b], non_blocking=True)
            down.wait_event(dec_done[b])
            h_od[b].copy_(o_dec[b], non_blocking=True)
            out_ready[b].record(down)

    def run(first, count):
        upload(first)
        for i in range(first, first + count):
            if i + 1 < first + count:
                upload(i + 1)
            compute_and_read_back(i)
            if i > first:  # the host takes each step's results one step behind the GPU
                out_ready[(i - 1) % 2].synchronize()
        out_ready[(first + count - 1) % 2].synchronize()

    run(0, warmup)
    torch.cuda.synchronize()
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(main)
    run(warmup, steps)
    t1.record(down)
    t1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return t0.elapsed_time(t1) * 1e-3, h2d, d2h


SPEC_M = 8  # tokens per verified draft window: the last accepted token + 7 drafts
# algorithmic bytes: verify reads the state once and, per token, q, k, v, z, b and writes
# o and the gate log (gk fp32, beta); fold reads and writes the state of every (sequence,
# head) with at least one accepted token and reads k, v, gk, beta of the accepted tokens
VERIFY_BYTES_PER_TOKEN = 3 * 2 * D + 4 * D + 4 + 4 * D + 4 * D + 4     # 2312
FOLD_BYTES_PER_TOKEN = 2 * 2 * D + 4 * D + 4                           # 1028


def run_speculative(steps, warmup, world, seed):
    """Speculative decoding on the decode workload's shape (256 sequences x 96 heads):
    verify of an SPEC_M-token window from the checkpoint, then the ReplaySSM fold of the
    accepted prefixes, whose lengths are drawn uniformly from 1..SPEC_M (mean 4.5; the
    pages report 2.6-4.7 accepted tokens per step)."""
    from linear_attention_serving_02_gb300 import kda

    N, H, m = DECODE_N, DECODE_H, SPEC_M
    wins = []
    for w in range(2):
        steps_in = [inputs.decode_step_inputs(N, H, seed=seed + 50 + w, step=t, device="cuda") for t in range(m)]
        win = {}
        for key in ("q", "k", "v", "z", "b"):
            x = torch.stack([st[key] for st in steps_in], dim=1)
            win[key] = x.reshape((N * m,) + tuple(x.shape[2:])).contiguous()
        win["A"] = steps_in[0]["A"]
        wins.append(win)
    state = inputs.decode_state(N, H, seed=seed + 60, device="cuda")
    g = torch.Generator().manual_seed(seed + 61)
    acc = torch.randint(1, m + 1, (N,), generator=g, dtype=torch.int32)
    acc_mean = float(acc.float().mean())
    acc = acc.cuda()
    o = torch.empty((N * m, H, D), dtype=torch.float32, device="cuda")
    gk = torch.empty((N * m, H, D), dtype=torch.float32, device="cuda")
    beta = torch.empty((N * m, H), dtype=torch.float32, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def one(i, ev=None):
        w = wins[i % 2]
        if ev:
            ev[0].record(stream)
        kda.kda_recurrent_verify(w["q"], w["k"], w["v"], w["z"], w["A"], w["b"], state, m, o=o, gk_log=gk,
                                 beta_log=beta)
        if ev:
            ev[1].record(stream)
        kda.kda_replay_fold(w["k"], w["v"], gk, beta, acc, state, m)
        if ev:
            ev[2].record(stream)

    for i in range(warmup):
        flush()
        one(i)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        one(warmup + j, evs[j])
    torch.cuda.synchronize()
    barrier(world)
    ver = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b, _ in evs) * 1e-3, world)
    fol = max_over_ranks(statistics.mean(b.elapsed_time(c) for _, b, c in evs) * 1e-3, world)
    pairs = N * H
    ver_bytes = pairs * (4 * D * D + m * VERIFY_BYTES_PER_TOKEN)
    fold_bytes = pairs * (2 * 4 * D * D + acc_mean * FOLD_BYTES_PER_TOKEN) + 4 * N
    return {"window": m, "accepted_mean": acc_mean, "sequences": N, "heads": H,
            "verify": {"ms": 1e3 * ver, "token_heads_per_s": world * pairs * m / ver,
                       "bytes_per_launch": ver_bytes, "achieved_gbs": ver_bytes / ver / 1e9},
            "fold": {"ms": 1e3 * fol, "bytes_per_launch": fold_bytes, "achieved_gbs": fold_bytes / fol / 1e9},
            "accepted_token_heads_per_s": world * pairs * acc_mean / (ver + fol),
            "finite": bool(torch.isfinite(state).all() and torch.isfinite(o).all())}


# fused decode: per (sequence, head) token the state read + write, x_q, x_k, x_v (bf16),
# the conv state read + write (3 streams x 3 inputs, bf16), z, b, g and y (fp32); the conv
# taps and the norm weight are read once per head
FUSED_BYTES_PER_TH = 2 * 4 * D * D + 3 * 2 * D + 2 * 9 * 2 * D + 4 * D + 4 + 4 * D + 4 * D   # 138500
FUSED_BYTES_PER_HEAD = 3 * D * 4 * 4


def run_fused_decode(steps, warmup, world, seed):
    """The fused decode layer step on the decode workload's shape (256 x 96, 1.6 GB state)."""
    from linear_attention_serving_02_gb300 import kda

    N, H = DECODE_N, DECODE_H
    prm = inputs.fused_decode_params(H, seed=seed + 70, device="cuda")
    pool = [inputs.fused_decode_step_inputs(N, H, seed=seed + 70, step=i, device="cuda") for i in range(4)]
    state = inputs.decode_state(N, H, seed=seed + 71, device="cuda")
    cs = torch.zeros((N, 3, 3, H, D), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((N, H, D), dtype=torch.float32, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def one(i):
        st = pool[i % len(pool)]
        kda.kda_fused_decode(st["x_q"], st["x_k"], st["x_v"], cs, prm["conv_w"], st["z"], st["A"], st["b"], st["g"],
                             prm["norm_w"], state, y=y)

    for i in range(warmup):
        flush()
        one(i)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        evs[j][0].record(stream)
        one(warmup + j)
        evs[j][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e-3, world)
    nbytes = N * H * FUSED_BYTES_PER_TH + H * FUSED_BYTES_PER_HEAD + 4 * D
    return {"sequences": N, "heads": H, "ms": 1e3 * t, "token_heads_per_s": world * N * H / t,
            "bytes_per_launch": nbytes, "achieved_gbs": nbytes / t / 1e9,
            "finite": bool(torch.isfinite(state).all() and torch.isfinite(y).all())}


def run_prefill_workload(which, steps, warmup, world, seed):
    """Prefill alone on one of the pages' prefill workloads, device-timed with CUDA events
    (bf16 o; inputs drawn on the device, so nothing here is oracle-checked: the parity
    tests cover these shapes):
      prefill one 8192-token sequence, 12 heads, initial state ~ N(0, 0.02^2);
      varlen  8 packed sequences of U[1024, 32768] tokens (from seed 0), 32 heads, zero
              initial states;
      long    one 1,048,576-token sequence, 12 heads, then 128 recurrent decode steps on its
              final state.
    Each timed call's inputs are larger than L2, so no flush runs between calls."""
    from linear_attention_serving_02_gb300 import kda

    if which == "prefill":
        H, T = PREFILL_H, PREFILL_T
        inp = inputs.prefill_inputs(T, H, 1, seed=seed, init_state=True, device="cuda")
        cu = cu_host = None
        n_seqs = 1
    elif which == "varlen":
        H = 32
        lens = inputs.varlen_lengths(8, 1024, 32768, seed=0)
        cu_host = inputs.cu_seqlens_from_lengths(lens)
        T = int(cu_host[-1])
        inp = inputs.prefill_inputs(T, H, len(lens), seed=seed, device="cuda")
        cu = cu_host.cuda()
        n_seqs = len(lens)
    else:
        H, T = 12, 1 << 20
        inp = inputs.prefill_inputs(T, H, 1, seed=seed, device="cuda")
        cu = cu_host = None
        n_seqs = 1
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, n_seqs, H), dtype=torch.uint8, device="cuda")
    o = torch.empty(inp["q"].shape, dtype=torch.bfloat16, device="cuda")
    S = torch.empty((n_seqs, H, D, D), dtype=torch.float32, device="cuda")
    main = torch.cuda.current_stream()

    def prefill():
        kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], initial_state=inp["S0"],
                              cu_seqlens=cu, cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws)

    for _ in range(warmup):
        prefill()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(steps):
        prefill()  # inputs of several GB: larger than L2, no flush needed
    e1.record(main)
    e1.synchronize()
    t = max_over_ranks(e0.elapsed_time(e1) * 1e-3 / steps, world)
    res = {"workload": which, "tokens": T, "heads": H, "sequences": n_seqs, "prefill_ms": 1e3 * t,
           "token_heads_per_s": world * T * H / t, "io_gbs": PREFILL_BYTES_PER_TH * T * H / t / 1e9}
    if which == "long":
        # the decode that follows: 128 steps of one token per head on the prefilled state
        dec = [inputs.decode_step_inputs(1, H, seed=seed + 5, step=i, device="cuda", A=inp["A"]) for i in range(8)]
        o_dec = torch.empty((1, H, D), dtype=torch.float32, device="cuda")
        def steps():
            for i in range(128):
                d = dec[i % len(dec)]
                kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["z"], d["A"], d["b"], S, o=o_dec)

        e0.record(main)
        steps()
        e1.record(main)
        e1.synchronize()
        res["decode_128_steps_ms"] = e0.elapsed_time(e1)
        # the same steps as one CUDA graph, as a serving loop replays its launch-bound decode
        # (each step launches one small kernel: the calls' host time dominates the loop above)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steps()
        graph.replay()
        torch.cuda.synchronize()
        e0.record(main)
        graph.replay()
        e1.record(main)
        e1.synchronize()
        res["decode_128_steps_graph_ms"] = e0.elapsed_time(e1)
        del graph
    res["finite"] = bool(torch.isfinite(S).all())
    del inp, ws, o, S
    torch.cuda.empty_cache()
    return res


def run_decode_only(steps, warmup, world, seed):
    """The decode step alone (256 sequences x 96 heads, 1.6 GB state updated in place), for
    kernel counters on a small process; L2 flushed between steps."""
    from linear_attention_serving_02_gb300 import kda

    state = inputs.decode_state(DECODE_N, DECODE_H, seed=seed + 1, device="cuda")
    dec = [inputs.decode_step_inputs(DECODE_N, DECODE_H, seed=seed + 1, step=i, device="cuda") for i in range(4)]
    o = torch.empty((DECODE_N, DECODE_H, D), dtype=torch.float32, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        flush()
        d = dec[i % len(dec)]
        kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["z"], d["A"], d["b"], state, o=o)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for j in range(steps):
        flush()
        d = dec[(warmup + j) % len(dec)]
        evs[j][0].record(stream)
        kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["z"], d["A"], d["b"], state, o=o)
        evs[j][1].record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e-3, world)
    nbytes = DECODE_BYTES_PER_TH * DECODE_N * DECODE_H
    return {"sequences": DECODE_N, "heads": DECODE_H, "ms": 1e3 * t, "achieved_gbs": nbytes / t / 1e9,
            "finite": bool(torch.isfinite(state).all())}


def prefill_roofline(res, hbm, tf_burst, peak_kind):
    """Roofline of a whole prefill call (all its kernels): the algorithmic bytes are its
    mandatory I/O (1540 B per token-head); the DRAM traffic is the per-token-head figure of
    the committed small-case capture (profiles/traffic.json, 8192 x 12) scaled to this
    call's token-heads, or null once the prefill kernels have changed since the capture."""
    th = res["tokens"] * res["heads"]
    t = res["prefill_ms"] * 1e-3
    gbs = PREFILL_BYTES_PER_TH * th / t / 1e9
    tfl = PREFILL_FLOPS_PER_TH * th / t / 1e12
    per_th = traffic_record(None, "kda_chunk_prefill")
    return {"kernel": "kda_chunk_prefill (all its kernels)", "bound": "hbm", "achieved": gbs, "peak": hbm,
            "unit": "GB/s", "frac": gbs / hbm, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": PREFILL_BYTES_PER_TH * th, "mma_tflops": tfl,
            "mma_frac_of_bf16": tfl / tf_burst, "traffic": None if per_th is None else per_th * th}


# ------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ------------------------------------------------------------------------------------
def oracle_sample(pre_cpu, prefill_heads, decode_pairs, seed=0):
    """Time the fp64 oracle on a sample: the prefill batch restricted to its first
    prefill_heads heads, plus decode_pairs (sequence, head) pairs of one decode token.
    Returns (seconds, token-heads processed, threads)."""
    import oracle

    h = prefill_heads
    sl = {k: (v[..., :h, :].contiguous() if k in ("q", "k", "v", "z") else v) for k, v in pre_cpu.items()}
    sl["b"] = pre_cpu["b"][..., :h].contiguous()
    sl["A"] = pre_cpu["A"][:h].contiguous()
    sl["S0"] = pre_cpu["S0"][:, :h].contiguous()
    P = decode_pairs
    st = inputs.decode_step_inputs(P, 1, seed=seed + 11)
    S0 = inputs.decode_state(P, 1, seed=seed + 12)
    threads = oracle.hardware_threads()
    t0 = time.perf_counter()
    oracle.kda_forward(sl["q"], sl["k"], sl["v"], sl["z"], sl["A"], sl["b"], S0=sl["S0"])
    oracle.kda_forward(st["q"].reshape(P, 1, 1, D), st["k"].reshape(P, 1, 1, D), st["v"].reshape(P, 1, 1, D),
                       st["z"].reshape(P, 1, 1, D), st["A"], st["b"].reshape(P, 1, 1), S0=S0)
    dt = time.perf_counter() - t0
    return dt, PREFILL_T * h + P, threads


def traffic_record(kernel_file, kernel_name):
    """DRAM bytes from a committed ncu summary (profiles/traffic.json), if it was taken on
    the current sources of that kernel (else None): bytes per launch for a kernel, bytes
    per token-head for the whole prefill."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_name)
        src = b""
        for fn in rec["sources"]:
            with open(os.path.join(ROOT, fn), "rb") as f:
                src += f.read()
        if hashlib.sha1(src).hexdigest() != rec["sources_sha1"]:
            return None
        key = "dram_bytes_per_launch" if "dram_bytes_per_launch" in rec else "dram_bytes_per_token_head"
        return float(rec[key])
    except Exception:
        return None


def main_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    pre_cpu = inputs.prefill_inputs(PREFILL_T, PREFILL_H, 1, seed=0, init_state=True)
    heads, pairs = 2, 1024
    for _ in range(args.warmup):
        oracle_sample(pre_cpu, heads, pairs)
    tot_s, tot_units, threads = 0.0, 0, 1
    for _ in range(args.steps):
        dt, units, threads = oracle_sample(pre_cpu, heads, pairs)
        tot_s += dt
        tot_units += units
    value = tot_units / tot_s
    sample = ("per step: prefill T=8192 restricted to %d of 12 heads (%d token-heads) + %d decode "
              "(sequence, head) pairs, one token each" % (heads, PREFILL_T * heads, pairs))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "token·head/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "token·head/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "token·head/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main_ours(args, rank, world, local):
    from linear_attention_serving_02_gb300 import kda

    hbm, tf_burst, tf_sust, peak_kind = peaks()
    pre_cpu, pre, state, dec = make_workload(rank)

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    t_wall = time.perf_counter()
    pre_ms, dec_ms, finite = run_ours_device(pre, state, dec, args.steps, args.warmup, world)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop() if clocks else None

    e2e_s, h2d, d2h = run_ours_e2e(pre_cpu, dec, args.steps, args.warmup, world)
    spec = run_speculative(max(1, min(args.steps, 50)), args.warmup, world, seed=1000 * rank)
    for part in ("verify", "fold"):
        spec[part]["frac_of_hbm"] = spec[part]["achieved_gbs"] / hbm
    fused = run_fused_decode(max(1, min(args.steps, 50)), args.warmup, world, seed=1000 * rank)
    fused["frac_of_hbm"] = fused["achieved_gbs"] / hbm
    # the pages' two larger prefill workloads, each on its own (a few calls: each is
    # milliseconds long and its inputs are many times larger than L2)
    pre_varlen = run_prefill_workload("varlen", max(1, min(args.steps, 5)), args.warmup, world, seed=1000 * rank)
    pre_varlen["roofline"] = prefill_roofline(pre_varlen, hbm, tf_burst, peak_kind)
    pre_long = run_prefill_workload("long", max(1, min(args.steps, 3)), args.warmup, world, seed=1000 * rank)
    pre_long["roofline"] = prefill_roofline(pre_long, hbm, tf_burst, peak_kind)

    pre_t = max_over_ranks(sum(pre_ms) / 1e3, world)
    dec_t = max_over_ranks(sum(dec_ms) / 1e3, world)
    step_t = max_over_ranks((sum(pre_ms) + sum(dec_ms)) / 1e3, world)
    e2e_t = max_over_ranks(e2e_s, world)
    K = args.steps
    th_pre = PREFILL_T * PREFILL_H
    th_dec = DECODE_N * DECODE_H
    units = world * K * (th_pre + th_dec)
    value = units / step_t

    # roofline of each part: algorithmic bytes (flops) per launch / average launch time
    pre_launch = pre_t / K
    dec_launch = dec_t / K
    dec_gbs = DECODE_BYTES_PER_TH * th_dec / dec_launch / 1e9
    pre_gbs = PREFILL_BYTES_PER_TH * th_pre / pre_launch / 1e9
    pre_tflops = PREFILL_FLOPS_PER_TH * th_pre / pre_launch / 1e12
    dec_traffic = traffic_record("linear_attention_serving_02_gb300/csrc/kda_decode.cu", "kda_decode_kernel<128>")
    roof_dec = {"kernel": "kda_decode_kernel<128>", "bound": "hbm", "achieved": dec_gbs, "peak": hbm, "unit": "GB/s",
                "frac": dec_gbs / hbm, "peak_kind": peak_kind + " (burst copy)",
                "traffic": dec_traffic, "algorithmic_bytes_per_launch": DECODE_BYTES_PER_TH * th_dec}
    pre_traffic = traffic_record(None, "kda_chunk_prefill")
    roof_pre = {"kernel": "kda_chunk_prefill (all its kernels)", "bound": "hbm", "achieved": pre_gbs,
                "peak": hbm, "unit": "GB/s", "frac": pre_gbs / hbm, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": PREFILL_BYTES_PER_TH * th_pre,
                "mma_tflops": pre_tflops, "mma_frac_of_bf16": pre_tflops / tf_burst,
                "traffic": None if pre_traffic is None else pre_traffic * th_pre}
    dominant = roof_dec if dec_t >= pre_t else roof_pre

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        dt, cu_units, reps = 0.0, 0, 0
        while dt < 10.0 or reps == 0:
            d1, u1, threads = oracle_sample(pre_cpu, PREFILL_H, 4096, seed=reps)
            dt += d1
            cu_units += u1
            reps += 1
        cpu = {"value": cu_units / dt, "unit": "token·head/s", "cores": threads, "kind": "oracle",
               "sample": "%d repetitions of: prefill B=1 T=8192 H=12 (all %d token-heads) + 4096 decode "
                         "(sequence, head) pairs, one token each; %.1f s of host time" % (reps, th_pre, dt)}
    line = {
        "metric": METRIC, "value": value, "unit": "token·head/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_t / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 operands split hi/lo, fp32 accumulate; decode f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": PREFILL_T,
                   "parallelism": "replicas x%d" % world, "l2": "device-timed steps: flushed between steps (512 MB write); e2e steps: working set (151 MB "
                         "of inputs, 1.6 GB of state) larger than L2"},
        "prefill": {"value": world * K * th_pre / pre_t, "unit": "token·head/s",
                    "tokens_per_s": world * K * PREFILL_T / pre_t, "ms": 1e3 * pre_launch, "roofline": roof_pre},
        "decode": {"value": world * K * DECODE_N / dec_t, "unit": "token/s (one per sequence)",
                   "token_heads_per_s": world * K * th_dec / dec_t, "ms": 1e3 * dec_launch, "roofline": roof_dec},
        "prefill_varlen": pre_varlen,
        "prefill_long": pre_long,
        "speculative": spec,
        "fused_decode": fused,
        "roofline": dominant,
        "cpu_baseline": cpu,
        "e2e": {"value": units / e2e_t, "unit": "token·head/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * (kda.kda_chunk_prefill_launch_count(PREFILL_T, 1, PREFILL_H) + 1),
        "clocks": clk,
        "outputs_finite": finite,
        "timed_wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--part", choices=["all", "speculative", "fused", "decode", "prefill", "varlen", "long"],
                    default="all",
                    help="'speculative' times only the verify + fold pair, 'fused' only the fused decode, "
                         "'decode' only the decode step (each 2-3 GB on the device; for profiling); "
                         "'prefill', 'varlen' and 'long' "
                         "time only the prefill of the 8192-token 12-head sequence (under 0.5 GB on the "
                         "device: the small case for kernel counters), of the packed 8 x U[1024, 32768] x "
                         "32-head batch and of the 1M-token sequence; each prints its object")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        main_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.part != "all":
            if args.part in ("prefill", "varlen", "long"):
                res = run_prefill_workload(args.part, args.steps, args.warmup, world, seed=1000 * rank)
            else:
                run = {"speculative": run_speculative, "fused": run_fused_decode, "decode": run_decode_only}[args.part]
                res = run(args.steps, args.warmup, world, seed=1000 * rank)
            if rank == 0:
                print(json.dumps({args.part: res}), flush=True)
            return
        main_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
