#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs, the
largest prefill workloads first, then the paged decode:
  * long causal prefill, B=1, H=16, Sq=Skv=8192, d=128;
  * the same with a 1024-key sliding window plus one sink key (key 0);
  * GQA causal prefill, B=2, Hq=32, Hkv=8, Sq=Skv=4096, d=128;
  * GQA varlen causal prefill, 8 packed sequences of seeded lengths in
    [256, 4096], Hq=32, Hkv=8, d=128;
  * paged split-KV decode, B=64, Hq=32, Hkv=8, d=128, 16-token pages,
    lengths uniform in [1024, 8192], 8 splits (split kernel + LSE merge).
Every call is bf16 in, fp32 accumulation, bf16 O and fp32 LSE out.

The headline ``value`` is the prefill forward throughput in TFLOP/s over the
four prefill calls: 4*B*Hq*Sq*Skv*d, halved for causal (the FLOP convention of
the pages' workloads), with exact visible (query, key) pairs x 4d for the
window and varlen calls.  Decode is reported as algorithmic KV bytes per
second beside it.  L2 is flushed (256 MB write, untimed) before every call.
Kernel times come from CUDA events recorded on the stream the kernels run on.

``--impl reference`` times the fp64 CPU oracle (the slow, obviously correct
program the kernels are checked against) on a bounded sample of the same
workload, on this host's cores.

``--gpus N`` with N > 1 and no torchrun environment re-launches this script
under ``torch.distributed.run`` with N processes (one per GPU); every rank
times its own replica of the workload and the slowest rank sets the time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % BF16 tensor peak; decode KV GB/s & % HBM peak"
UNIT = "TFLOP/s"
WORKLOAD = ("long causal prefill B=1 H=16 S=8192 d=128 (+ window W=1024 with 1 sink key) + "
            "GQA causal prefill B=2 Hq=32 Hkv=8 S=4096 d=128 (+ varlen 8 seqs L~U[256,4096]) + "
            "paged decode B=64 Hq=32 Hkv=8 d=128 L~U[1024,8192] page=16 splits=8; bf16")
L2_FLUSH_BYTES = 256 << 20
BM = 128                 # query rows per tile in the kernels (the re-read model's Bm)
EX2_PER_CLK_SM = 32      # ex2.approx results per clock per SM, measured on this GPU
NUM_SMS = 152


# ------------------------------------------------------------------ accounting

def prefill_flops(B, H, Sq, Skv, d, causal):
    """The workloads' FLOP convention: 4*B*H*Sq*Skv*d, halved when causal."""
    f = 4.0 * B * H * Sq * Skv * d
    return f / 2 if causal else f


def row_pairs(i, Lq, Lk, causal, window=0, n_sink=0):
    """Keys query row i of a (Lq, Lk) sequence sees: key j is visible iff
    j < Lk and, when causal, j <= i + (Lk - Lq) (bottom-right alignment), and,
    with a window W > 0, also j > i + (Lk - Lq) - W or j < n_sink."""
    off = Lk - Lq
    hi = min(i + off, Lk - 1) if causal else Lk - 1
    if hi < 0:
        return 0
    if window <= 0:
        return hi + 1
    lo = i + off - window                 # window keys are those in (lo, hi]
    return hi - max(lo, -1) + max(0, min(n_sink, lo + 1, hi + 1))


def visible_pairs(Lq, Lk, causal, window=0, n_sink=0):
    """Exact number of (query, key) pairs one head of one sequence computes."""
    return sum(row_pairs(i, Lq, Lk, causal, window, n_sink) for i in range(Lq))


def decode_kv_bytes(seqlens, Hkv, d):
    """Algorithmic bytes of one decode call: every visible key and value once."""
    return int(sum(int(L) for L in seqlens)) * Hkv * d * 2 * 2


def reread_model_bytes(B, Hq, Hkv, Sq, Skv, d, q_tiles_per_kv=None):
    """The pages' fused-kernel HBM traffic model: Q and O once, K and V once
    per 128-row query tile ((Q + O) + (K + V) * ceil(Sq / Bm)), bf16."""
    tiles = q_tiles_per_kv if q_tiles_per_kv is not None else -(-Sq // BM) * (Hq // Hkv)
    return 2 * (2 * B * Sq * Hq * d) + 2 * (2 * B * Skv * Hkv * d) * tiles


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash(name):
    with open(os.path.join(ROOT, "exact_attention_08_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file, summary):
    """DRAM bytes per launch recorded from an ncu capture of the same kernel
    source (profiles/traffic.json); None when absent or the kernel changed."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(summary)
    if not e or e.get("source_sha256_16") != kernel_source_hash(kernel_file):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        with open(self.out.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            c = [x.strip() for x in l.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                smax.append(float(c[2]))
            except ValueError:
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity on one
    process).  This is the only cross-rank step of the bench: every rank runs
    its own copy of the workload (weak scaling) and the slowest rank sets the
    time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def launch_ranks(args, argv):
    """Runs this script under torch.distributed.run with args.gpus processes on
    this node (rendezvous on 127.0.0.1) and returns its exit code.  Rank 0
    prints the JSON line; the per-rank device is LOCAL_RANK."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1",
           f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def init_ranks(backend, device=None):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)
    return world, rank, local


def finish_ranks(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_stub(args):
    """The rank harness with a CPU stand-in for the kernels (gloo): each rank
    'processes' a fixed number of units by sleeping, and the line is formed
    exactly as for the real run (max over ranks, whole-job value).  Used by
    the multi-process CPU test of the launch path."""
    world, rank, _ = init_ranks("gloo")
    units_per_step = 1.0e12
    for _ in range(args.warmup):
        time.sleep(0.001)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep(0.002 * (1 + rank))
    sec = time.perf_counter() - t0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    (sec_max,) = max_over_ranks([sec])
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": world * args.steps * units_per_step / sec_max / 1e12,
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec_max * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "stub": True, "rank_seconds_max": sec_max}))
    finish_ranks(world)


# ------------------------------------------------------------------ workloads

def prefill_workloads():
    """The four prefill calls of a step: (name, inputs, FLOPs, visible pairs,
    FLOPs in the causal convention)."""
    import workloads
    out = []
    for name, x in (("long_causal_s8192", workloads.long_causal(False)),
                    ("long_window1024_sink1_s8192", workloads.long_causal(True)),
                    ("gqa_causal_s4096", workloads.gqa_causal()),
                    ("gqa_varlen_8seq", workloads.gqa_varlen())):
        if hasattr(x, "cu_q"):
            lq = (x.cu_q[1:] - x.cu_q[:-1]).tolist()
            lk = (x.cu_k[1:] - x.cu_k[:-1]).tolist()
            Hq, d = x.q.shape[1], x.q.shape[2]
            pairs = Hq * sum(visible_pairs(a, b, x.causal, x.window, x.n_sink)
                             for a, b in zip(lq, lk))
            conv = sum(prefill_flops(1, Hq, a, b, d, x.causal) for a, b in zip(lq, lk))
            flops = 4.0 * d * pairs
        else:
            B, Sq, Hq, d = x.q.shape
            Skv = x.k.shape[1]
            pairs = B * Hq * visible_pairs(Sq, Skv, x.causal, x.window, x.n_sink)
            conv = prefill_flops(B, Hq, Sq, Skv, d, x.causal)
            flops = 4.0 * d * pairs if x.window > 0 else conv
        out.append((name, x, flops, pairs, conv))
    return out


# ------------------------------------------------------------------ CPU oracle timings

def _oracle_rows(S, stride):
    import numpy as np
    return np.arange(0, S, stride, dtype=np.int32)


def oracle_prefill_sample(pre, stride, heads=None):
    """Times the oracle on every stride-th query row of each prefill call
    (all heads, or the first `heads` query heads).  Returns a list of
    (call name, visible-pair FLOPs of the sample, seconds)."""
    import oracle
    out = []
    for name, x, _, _, _ in pre:
        flops, sec = 0.0, 0.0
        varlen = hasattr(x, "cu_q")
        Hq, d = x.q.shape[-2], x.q.shape[-1]
        Hkv = x.k.shape[-2]
        hq = heads or Hq
        hk = max(1, -(-hq // (Hq // Hkv)))
        if varlen:
            cq, ck = x.cu_q.tolist(), x.cu_k.tolist()
            seqs = [(x.q[None, cq[s]:cq[s + 1]], x.k[None, ck[s]:ck[s + 1]],
                     x.v[None, ck[s]:ck[s + 1]]) for s in range(len(cq) - 1)]
        else:
            seqs = [(x.q, x.k, x.v)]
        for q, k, v in seqs:
            B, Sq, Skv = q.shape[0], q.shape[1], k.shape[1]
            rows = _oracle_rows(Sq, stride)
            qn = q[:, :, :hq].double().numpy()
            kn = k[:, :, :hk].double().numpy()
            vn = v[:, :, :hk].double().numpy()
            t0 = time.perf_counter()
            oracle.attn_fwd(qn, kn, vn, x.scale, x.causal, x.window, x.n_sink, rows=rows)
            sec += time.perf_counter() - t0
            flops += 4.0 * d * B * hq * sum(row_pairs(int(r), Sq, Skv, x.causal, x.window,
                                                      x.n_sink) for r in rows)
        out.append((name, flops, sec))
    return out


def cpu_baseline(pre, dx):
    """The oracle as it stands, on this host's cores, on a bounded sample of
    the step (every other query row of every prefill call and head, and 8
    requests of the decode), in the line's units; plus a single-thread run of
    the tiny configuration."""
    import oracle
    import workloads
    stride = 2
    parts = oracle_prefill_sample(pre, stride)
    flops, sec = sum(p[1] for p in parts), sum(p[2] for p in parts)
    full = {name: fl for name, _, fl, _, _ in pre}
    per_call = {name: {"tflops": f / s / 1e12, "sample_seconds": s,
                       "full_call_seconds_est": s * full[name] / f}
                for name, f, s in parts}
    req = list(range(8))
    k, v = dx.contiguous_kv(req)
    t0 = time.perf_counter()
    oracle.attn_decode(dx.q[req].double().numpy(), k.double().numpy(), v.double().numpy(),
                       dx.seqlens[req].numpy(), dx.scale)
    dsec = time.perf_counter() - t0
    dbytes = decode_kv_bytes(dx.seqlens[req].tolist(), dx.k_pages.shape[2], dx.k_pages.shape[3])
    cores = oracle.num_threads()
    tiny = workloads.tiny_mha()
    prev = oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        reps = 20
        for _ in range(reps):
            oracle.attn_fwd(tiny.q.double().numpy(), tiny.k.double().numpy(),
                            tiny.v.double().numpy(), tiny.scale)
        tsec = (time.perf_counter() - t0) / reps
    finally:
        oracle.set_num_threads(prev)
    return {"value": flops / sec / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": sec,
            "sample": "every other query row of every head of the four prefill calls "
                      "(visible-pair FLOPs of those rows)",
            "per_call": per_call,
            "decode": {"value": dbytes / dsec / 1e9, "unit": "GB/s", "seconds": dsec,
                       "sample": "requests 0-7 of the decode batch"},
            "single_thread_tiny": {"ms": tsec * 1e3,
                                   "tflops": prefill_flops(1, 1, 128, 128, 64, False) / tsec / 1e12,
                                   "workload": "B=1 H=1 S=128 d=64 non-causal, 1 thread"}}


def run_reference(args):
    """The oracle (fp64, CPU) as the reference arm: each step a bounded sample
    of the step's prefill calls (every 16th query row of query heads 0-1 of
    each call), on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    pre = prefill_workloads()
    stride, heads = 16, 2
    for _ in range(args.warmup):
        oracle_prefill_sample(pre, stride, heads)
    fl, t = 0.0, []
    for _ in range(args.steps):
        parts = oracle_prefill_sample(pre, stride, heads)
        fl = sum(p[1] for p in parts)
        t.append(sum(p[2] for p in parts))
    sec = statistics.median(t)
    val = fl / sec / 1e12
    sample = ("every 16th query row of query heads 0-1 of each of the four prefill calls "
              "(visible-pair FLOPs of those rows)")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------------ the GPU run

def timed_calls(stream, flush, fn, n=20, warm=3, tag=1):
    """Median CUDA-event time (ms) of fn() over n calls after warm calls, L2
    flushed before each."""
    import torch
    ts = []
    for it in range(n + warm):
        with torch.cuda.stream(stream):
            flush.fill_(tag)
            a, b = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            a.record(stream)
            fn()
            b.record(stream)
        if it >= warm:
            ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the timed variants outside the step")
    ap.add_argument("--stub", action="store_true",
                    help="CPU stand-in for the kernels (tests of the rank harness)")
    argv = sys.argv[1:]
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_ranks(args, argv)
    if args.stub:
        return run_stub(args)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import exact_attention_08_gb300 as ea
    import workloads

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_ranks("nccl", dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # ---------------------------------------------------------------- inputs (resident)
    pre = prefill_workloads()
    calls = []   # (name, fn, device inputs, device outputs)
    for name, x, flops, pairs, conv in pre:
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        if hasattr(x, "cu_q"):
            cq, ck = x.cu_q.to(dev), x.cu_k.to(dev)
            lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=dev)

            def fn(q=q, k=k, v=v, o=o, lse=lse, cq=cq, ck=ck, x=x):
                ea.attn_fwd_ex(q, k, v, cq, ck, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k,
                               o=o, lse=lse, causal=x.causal, window=x.window,
                               n_sink=x.n_sink, scale=x.scale, stream=stream)
            ins = (q, k, v, cq, ck)
        else:
            lse = torch.empty(q.shape[0], q.shape[2], q.shape[1], dtype=torch.float32,
                              device=dev)

            def fn(q=q, k=k, v=v, o=o, lse=lse, x=x):
                ea.attn_fwd_ex(q, k, v, o=o, lse=lse, causal=x.causal, window=x.window,
                               n_sink=x.n_sink, scale=x.scale, stream=stream)
            ins = (q, k, v)
        calls.append((name, fn, ins, (o, lse)))
    dx = workloads.paged_decode()
    dq, dkp, dvp = dx.q.to(dev), dx.k_pages.to(dev), dx.v_pages.to(dev)
    dpt, dsl = dx.page_table.to(dev), dx.seqlens.to(dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[0], dq.shape[1], dtype=torch.float32, device=dev)
    Hkv_d, d_d = dx.k_pages.shape[2], dx.k_pages.shape[3]
    dws = torch.empty(ea.attn_decode_workspace_size(dq.shape[0], dq.shape[1], d_d,
                                                    dx.num_splits),
                      dtype=torch.uint8, device=dev)

    def decode_fn(q=dq, pt=dpt, sl=dsl, o=do, lse=dlse):
        ea.attn_decode_paged(q, dkp, dvp, pt, sl, o, lse, num_splits=dx.num_splits,
                             scale=dx.scale, workspace=dws, stream=stream)

    flops = [c[2] for c in pre]
    pairs_total = sum(c[3] for c in pre)
    kv_bytes = decode_kv_bytes(dx.seqlens.tolist(), Hkv_d, d_d)
    n_calls = len(calls) + 1
    # the four forward launches, and the decode's request order, split and merge
    launches_per_step = len(calls) + 3

    def step(ev):
        with torch.cuda.stream(stream):
            for c, (_, fn, _, _) in enumerate(calls):
                flush.fill_(c + 1)
                ev[2 * c].record(stream)
                fn()
                ev[2 * c + 1].record(stream)
            flush.fill_(9)
            ev[2 * len(calls)].record(stream)
            decode_fn()
            ev[2 * len(calls) + 1].record(stream)

    def mk():
        return [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_calls)]

    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize(dev)
    if ea.attn_device_status(stream) != ea.ATTN_OK:
        raise RuntimeError("device status reported an error during warm-up")

    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    evs = [mk() for _ in range(args.steps)]
    wall0 = time.perf_counter()
    for ev in evs:
        step(ev)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop()
    status = ea.attn_device_status(stream)
    if status != ea.ATTN_OK:
        raise RuntimeError(f"device status {ea.attn_status_string(status)}")

    K = args.steps
    per_call = [[e[2 * c].elapsed_time(e[2 * c + 1]) for e in evs] for c in range(n_calls)]
    sums = [sum(t) for t in per_call]
    sums = max_over_ranks(sums, dev)
    tot_pre = sum(sums[:-1])
    tot_dec = sums[-1]
    value = world * K * sum(flops) / (tot_pre / 1e3) / 1e12
    dec_gbs = world * K * kv_bytes / (tot_dec / 1e3) / 1e9
    hbm, bf16, src = peaks()

    # ---------------------------------------------------------------- end to end (host buffers)
    # Pipelined like a serving loop over the same calls: host->device copies
    # of the next call's inputs, this call's kernels and device->host copies
    # of the previous call's outputs run on three streams over double-
    # buffered device tensors; every copy of every timed step stays inside
    # the timed region.  Prefill inputs are q, k, v (and the varlen offsets);
    # decode inputs are the new queries, the page table and the lengths (the
    # KV cache is device-resident state that earlier steps wrote).
    e2e_steps = max(3, min(10, K))
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    jobs = []  # (host inputs, [device input copies x2], [device outputs x2], launcher)
    for name, fn, ins, outs in calls:
        x = next(p[1] for p in pre if p[0] == name)
        h_in = [t.cpu().pin_memory() for t in ins]
        d_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
        d_out = [[torch.empty_like(t) for t in outs] for _ in range(2)]
        h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
        if hasattr(x, "cu_q"):
            def launch(di, dout, x=x):
                q, k, v, cq, ck = di
                ea.attn_fwd_ex(q, k, v, cq, ck, max_seqlen_q=x.max_q, max_seqlen_k=x.max_k,
                               o=dout[0], lse=dout[1], causal=x.causal, window=x.window,
                               n_sink=x.n_sink, scale=x.scale, stream=stream)
        else:
            def launch(di, dout, x=x):
                q, k, v = di
                ea.attn_fwd_ex(q, k, v, o=dout[0], lse=dout[1], causal=x.causal,
                               window=x.window, n_sink=x.n_sink, scale=x.scale, stream=stream)
        jobs.append(("prefill", h_in, d_in, d_out, h_out, launch))
    d_ins = (dq, dpt, dsl)
    h_in = [t.cpu().pin_memory() for t in d_ins]

    def dlaunch(di, dout):
        q, pt, sl = di
        ea.attn_decode_paged(q, dkp, dvp, pt, sl, dout[0], dout[1], num_splits=dx.num_splits,
                             scale=dx.scale, workspace=dws, stream=stream)
    jobs.append(("decode", h_in, [[torch.empty_like(t) for t in d_ins] for _ in range(2)],
                 [[torch.empty_like(t) for t in (do, dlse)] for _ in range(2)],
                 [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (do, dlse)],
                 dlaunch))
    ev_in = {}
    ev_comp = {}
    ev_out = {}

    def e2e_run(kind, t):
        b = t % 2
        for j, (knd, hi, di, dout, ho, launch) in enumerate(jobs):
            if knd != kind:
                continue
            key = (j, b)
            with torch.cuda.stream(s_in):
                if key in ev_comp:
                    s_in.wait_event(ev_comp[key])   # the kernel that read this buffer
                for src, dst in zip(hi, di[b]):
                    dst.copy_(src, non_blocking=True)
                ev_in[key] = torch.cuda.Event()
                ev_in[key].record(s_in)
            stream.wait_event(ev_in[key])
            if key in ev_out:
                stream.wait_event(ev_out[key])      # its outputs have been read back
            launch(di[b], dout[b])
            ev_comp[key] = torch.cuda.Event()
            ev_comp[key].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[key])
                for src, dst in zip(dout[b], ho):
                    dst.copy_(src, non_blocking=True)
                ev_out[key] = torch.cuda.Event()
                ev_out[key].record(s_out)

    def e2e_time(kind):
        for t in range(2):
            e2e_run(kind, t)
        torch.cuda.synchronize(dev)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for t in range(e2e_steps):
            e2e_run(kind, t)
        s_in.wait_stream(s_out)
        e1.record(s_in)
        torch.cuda.synchronize(dev)
        return max_over_ranks([e0.elapsed_time(e1)], dev)[0]

    def nbytes(ts):
        return sum(t.numel() * t.element_size() for t in ts)

    e2e_pre_ms = e2e_time("prefill")
    e2e_dec_ms = e2e_time("decode")
    if ea.attn_device_status(stream) != ea.ATTN_OK:
        raise RuntimeError("device status reported an error in the end-to-end calls")
    pre_h2d = sum(nbytes(j[1]) for j in jobs if j[0] == "prefill")
    pre_d2h = sum(nbytes(j[4]) for j in jobs if j[0] == "prefill")
    dec_h2d = sum(nbytes(j[1]) for j in jobs if j[0] == "decode")
    dec_d2h = sum(nbytes(j[4]) for j in jobs if j[0] == "decode")
    e2e_val = world * e2e_steps * sum(flops) / (e2e_pre_ms / 1e3) / 1e12
    e2e_dec = world * e2e_steps * kv_bytes / (e2e_dec_ms / 1e3) / 1e9

    variants = {} if args.no_variants else run_variants(ea, workloads, dev, stream, flush)
    if ea.attn_device_status(stream) != ea.ATTN_OK:
        raise RuntimeError("device status reported an error in the variants")

    if rank == 0:
        achieved = sum(flops) * K / (tot_pre / 1e3) / 1e12
        dec_achieved = kv_bytes * K / (tot_dec / 1e3) / 1e9
        tr = profiled_traffic("attn_fwd_sm103.cu", "attn_fwd_step_prefill_calls")
        dtr = profiled_traffic("attn_decode_sm103.cu", "attn_decode_split_b64hq32hkv8d128")
        sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
        ex2_peak = EX2_PER_CLK_SM * NUM_SMS * sm_mhz * 1e6
        per = {}
        for c, (name, x, fl, pairs, conv) in enumerate(pre):
            ms = statistics.median(per_call[c])
            per[name] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12,
                         "frac": fl / (ms / 1e3) / 1e12 / bf16, "flops": fl,
                         "visible_pairs": pairs, "causal_convention_flops": conv}
        unique = 0
        model = 0
        for name, x, *_ in pre:
            if hasattr(x, "cu_q"):
                lq = (x.cu_q[1:] - x.cu_q[:-1]).tolist()
                Hq, d = x.q.shape[1], x.q.shape[2]
                Hkv = x.k.shape[1]
                unique += sum(2 * L * d * (2 * Hq + 2 * Hkv) + 4 * L * Hq for L in lq)
                model += sum(reread_model_bytes(1, Hq, Hkv, L, L, d) for L in lq)
            else:
                B, Sq, Hq, d = x.q.shape
                Skv, Hkv = x.k.shape[1], x.k.shape[2]
                unique += 2 * B * d * (2 * Sq * Hq + 2 * Skv * Hkv) + 4 * B * Hq * Sq
                model += reread_model_bytes(B, Hq, Hkv, Sq, Skv, d)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": (tot_pre + tot_dec) / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "prefill_flops_per_step": sum(flops),
                       "decode_kv_bytes_per_step": kv_bytes,
                       "l2": "flushed before every call (256 MB write, untimed)",
                       "parallelism": f"replicas x{world} (each rank its own copy)"},
            "prefill": per,
            "decode": {"value": dec_gbs, "unit": "GB/s", "ms": statistics.median(per_call[-1]),
                       "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": hbm,
                                    "unit": "GB/s", "frac": dec_achieved / hbm,
                                    "peak_source": src, "traffic": dtr}},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16,
                         "unit": "TFLOP/s", "frac": achieved / bf16, "peak_source": src,
                         "traffic": tr, "kernel": "attn_fwd_kernel<128>",
                         "launches_per_step": len(calls)},
            "secondary_ceilings": {
                "exp2": {"achieved_per_s": pairs_total * K / (tot_pre / 1e3),
                         "peak_per_s": ex2_peak,
                         "frac": pairs_total * K / (tot_pre / 1e3) / ex2_peak,
                         "note": "one exponential per visible pair; peak = 32 ex2.approx per "
                                 "clock per SM (measured) x 152 SMs x median SM clock"},
                "hbm_bytes": {"unique_bytes_per_step": unique,
                              "reread_model_bytes_per_step": model,
                              "measured_dram_bytes_per_step": tr,
                              "model_gbs_at_measured_time": model * K / (tot_pre / 1e3) / 1e9,
                              "peak_gbs": hbm,
                              "note": "(Q+O) + (K+V) x ceil(Sq/128) per KV head group, as if "
                                      "no K/V tile were reused through L2"}},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": pre_h2d + dec_h2d,
                    "d2h_bytes_per_step": pre_d2h + dec_d2h, "steps": e2e_steps,
                    "prefill_ms_per_step": e2e_pre_ms / e2e_steps,
                    "decode": {"value": e2e_dec, "unit": "GB/s",
                               "ms_per_step": e2e_dec_ms / e2e_steps,
                               "h2d_bytes_per_step": dec_h2d, "d2h_bytes_per_step": dec_d2h,
                               "note": "new queries, page table and lengths in; O and LSE "
                                       "out; the KV cache stays resident"}},
            "gpu_launches": launches_per_step * K,
            "clocks": clocks,
            "variants": variants,
            "wall_s_timed": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(pre, dx)
        print(json.dumps(line))
    finish_ranks(world)


def run_variants(ea, workloads, dev, stream, flush):
    """Paths timed apart from the step (not part of `value`), each on its own
    workload, 20 calls after 3 warm-up calls with L2 flushed before each."""
    import torch
    out = {}
    # prefill MHA, B=4 H=16 S=2048 d=128: non-causal, causal, and with logit sinks
    x2 = {c: workloads.prefill_mha(c) for c in (False, True)}
    dev2 = {c: (x.q.to(dev), x.k.to(dev), x.v.to(dev)) for c, x in x2.items()}
    o2 = torch.empty_like(dev2[False][0])
    l2 = torch.empty(4, 16, 2048, dtype=torch.float32, device=dev)
    r = {}
    for c, (q, k, v) in dev2.items():
        ms = timed_calls(stream, flush, lambda q=q, k=k, v=v, c=c: ea.attn_fwd(
            q, k, v, o2, l2, causal=c, scale=x2[c].scale, stream=stream))
        fl = prefill_flops(4, 16, 2048, 2048, 128, c)
        r["causal" if c else "noncausal"] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12}
    out["prefill_mha_b4h16s2048d128"] = r
    q, k, v = dev2[False]
    sink = workloads.logit_sinks(2101, 16).to(dev)
    ms = timed_calls(stream, flush, lambda: ea.attn_fwd_ex_sink(
        q, k, v, sink, o=o2, lse=l2, causal=False, scale=x2[False].scale, stream=stream))
    out["logit_sink_prefill_noncausal_b4h16s2048"] = {
        "ms": ms, "tflops": prefill_flops(4, 16, 2048, 2048, 128, False) / (ms / 1e3) / 1e12}
    # the same non-causal prefill with BHSD-stored q, k, v and o
    qb, kb, vb = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
    ob = torch.empty_like(qb)
    ms = timed_calls(stream, flush, lambda: ea.attn_fwd_strided(
        qb, kb, vb, ob, l2, causal=False, scale=x2[False].scale, stream=stream))
    out["prefill_noncausal_bhsd_b4h16s2048"] = {
        "ms": ms, "tflops": prefill_flops(4, 16, 2048, 2048, 128, False) / (ms / 1e3) / 1e12}
    del qb, kb, vb, ob
    # decode with logit sinks
    dx = workloads.paged_decode()
    dq, dkp, dvp = dx.q.to(dev), dx.k_pages.to(dev), dx.v_pages.to(dev)
    dpt, dsl = dx.page_table.to(dev), dx.seqlens.to(dev)
    do = torch.empty_like(dq)
    dl = torch.empty(64, 32, dtype=torch.float32, device=dev)
    dws = torch.empty(ea.attn_decode_workspace_size(64, 32, 128, 8), dtype=torch.uint8,
                      device=dev)
    sink_d = workloads.logit_sinks(5101, 32).to(dev)
    ms = timed_calls(stream, flush, lambda: ea.attn_decode_paged_sink(
        dq, dkp, dvp, dpt, dsl, sink_d, do, dl, num_splits=8, scale=dx.scale, workspace=dws,
        stream=stream))
    kvb = decode_kv_bytes(dx.seqlens.tolist(), 8, 128)
    out["logit_sink_decode_b64hq32hkv8"] = {"ms": ms, "kv_gbs": kvb / (ms / 1e3) / 1e9}
    del dq, dkp, dvp, dpt, dsl, do, dl, dws
    # chunked prefill on a paged cache (512-row query blocks at the end of
    # 2048-8192-key caches)
    cx = workloads.chunked_prefill()
    cc = cx.cache
    cq, ckp, cvp = cx.q.to(dev), cc.k_pages.to(dev), cc.v_pages.to(dev)
    cpt, ccu, csl = cc.page_table.to(dev), cx.cu_q.to(dev), cc.seqlens.to(dev)
    co = torch.empty_like(cq)
    cl = torch.empty(cq.shape[1], cq.shape[0], dtype=torch.float32, device=dev)
    lqs = (cx.cu_q[1:] - cx.cu_q[:-1]).tolist()
    lks = cc.seqlens.tolist()
    c_pairs = sum(visible_pairs(a, b, True) for a, b in zip(lqs, lks))
    c_flops = 4.0 * cq.shape[2] * cq.shape[1] * c_pairs
    ms = timed_calls(stream, flush, lambda: ea.attn_fwd_paged(
        cq, ckp, cvp, cpt, ccu, csl, co, cl, max_seqlen_q=cx.max_q, causal=True,
        scale=cx.scale, stream=stream))
    out["chunked_prefill_paged_b8hq32hkv8"] = {
        "workload": "B=8 Hq=32 Hkv=8 d=128, caches of 2048-8192 keys in 16-key pages, the last "
                    "512 tokens as the causal query block",
        "ms": ms, "flops": c_flops, "tflops": c_flops / (ms / 1e3) / 1e12}
    del cq, ckp, cvp, cpt, ccu, csl, co, cl
    # backward of the prefill MHA calls (same inputs, dO ~ N(0,1))
    gout = workloads.grad_output(7001, dev2[False][0].shape).to(dev)
    bws = torch.empty(ea.attn_bwd_workspace_size(4, 16, 2048), dtype=torch.uint8, device=dev)
    bw = {}
    for c, (q, k, v) in dev2.items():
        o = torch.empty_like(q)
        lse = torch.empty(4, 16, 2048, dtype=torch.float32, device=dev)
        ea.attn_fwd(q, k, v, o, lse, causal=c, scale=x2[c].scale, stream=stream)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ms = timed_calls(stream, flush, lambda q=q, k=k, v=v, o=o, lse=lse, c=c: ea.attn_bwd(
            q, k, v, o, lse, gout, gq, gk, gv, causal=c, scale=x2[c].scale, workspace=bws,
            stream=stream), n=10)
        fl = 2.5 * prefill_flops(4, 16, 2048, 2048, 128, c)
        bw["causal" if c else "noncausal"] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12}
    bw["note"] = "FLOPs 2.5x the forward's (five products)"
    out["backward_b4h16s2048d128"] = bw
    # head dimension 256: the forward, then the backward of its output
    d256, b256 = {}, {}
    for c in (False, True):
        xd = workloads.dense_inputs(7101 + int(c), 4, 16, 16, 2048, 2048, 256, c)
        qd, kd, vd = xd.q.to(dev), xd.k.to(dev), xd.v.to(dev)
        od = torch.empty_like(qd)
        ld = torch.empty(4, 16, 2048, dtype=torch.float32, device=dev)
        ms = timed_calls(stream, flush, lambda: ea.attn_fwd(
            qd, kd, vd, od, ld, causal=c, scale=xd.scale, stream=stream))
        fl = prefill_flops(4, 16, 2048, 2048, 256, c)
        d256["causal" if c else "noncausal"] = {"ms": ms, "tflops": fl / (ms / 1e3) / 1e12}
        gd = workloads.grad_output(7111 + int(c), qd.shape).to(dev)
        gq, gk, gv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ms = timed_calls(stream, flush, lambda: ea.attn_bwd(
            qd, kd, vd, od, ld, gd, gq, gk, gv, causal=c, scale=xd.scale, workspace=bws,
            stream=stream), n=10)
        b256["causal" if c else "noncausal"] = {"ms": ms, "tflops": 2.5 * fl / (ms / 1e3) / 1e12}
        del qd, kd, vd, od, ld, gd, gq, gk, gv
    out["prefill_d256_b4h16s2048"] = d256
    b256["note"] = ("FLOPs 2.5x the forward's (five products); dV, dK and dQ from three "
                    "launches, each recomputing the scores")
    out["backward_d256_b4h16s2048"] = b256
    # head dimension 256 on a paged cache: the decode (the decode workload's
    # shape) and chunked prefill (the chunked-prefill workload's shape)
    dx = workloads.paged_decode_inputs(5301, 64, 32, 8, 256, 1024, 8192, num_splits=8)
    dq, dkp, dvp, dpt, dsl = (t.to(dev) for t in (dx.q, dx.k_pages, dx.v_pages, dx.page_table,
                                                  dx.seqlens))
    do = torch.empty_like(dq)
    dl = torch.empty(64, 32, dtype=torch.float32, device=dev)
    dws = torch.empty(ea.attn_decode_workspace_size(64, 32, 256, 8), dtype=torch.uint8,
                      device=dev)
    ms = timed_calls(stream, flush, lambda: ea.attn_decode_paged(
        dq, dkp, dvp, dpt, dsl, do, dl, num_splits=8, scale=dx.scale, workspace=dws,
        stream=stream))
    kvb = decode_kv_bytes(dx.seqlens.tolist(), 8, 256)
    out["decode_d256_b64hq32hkv8"] = {"ms": ms, "kv_gbs": kvb / (ms / 1e3) / 1e9,
                                      "kv_bytes": kvb}
    del dq, dkp, dvp, dpt, dsl, do, dl, dws
    cx = workloads.paged_prefill_inputs(6301, 8, 32, 8, 256, 2048, 8192, 512, 512)
    cc = cx.cache
    cq, ckp, cvp, cpt, ccu, csl = (t.to(dev) for t in (cx.q, cc.k_pages, cc.v_pages,
                                                       cc.page_table, cx.cu_q, cc.seqlens))
    co = torch.empty_like(cq)
    cl = torch.empty(cq.shape[1], cq.shape[0], dtype=torch.float32, device=dev)
    lqs = (cx.cu_q[1:] - cx.cu_q[:-1]).tolist()
    c_flops = 4.0 * 256 * 32 * sum(visible_pairs(a, b, True)
                                   for a, b in zip(lqs, cc.seqlens.tolist()))
    ms = timed_calls(stream, flush, lambda: ea.attn_fwd_paged(
        cq, ckp, cvp, cpt, ccu, csl, co, cl, max_seqlen_q=cx.max_q, causal=True,
        scale=cx.scale, stream=stream))
    out["chunked_prefill_paged_d256_b8hq32hkv8"] = {"ms": ms, "flops": c_flops,
                                                    "tflops": c_flops / (ms / 1e3) / 1e12}
    del cq, ckp, cvp, cpt, ccu, csl, co, cl
    torch.cuda.synchronize(dev)
    return out


if __name__ == "__main__":
    sys.exit(main() or 0)
