#!/usr/bin/env python
"""Benchmark of batched paged-KV context attention on GB300.

Workload: the Llama-3-8B-shaped prefill (batch 8, q_len = kv_len ~ U[512, 2048],
32 query heads / 8 kv heads, head_dim 128, page_size 32, HND, bf16 N(0,1),
pages scattered over a pool twice the needed size, causal), drawn by
workload.config(2) with seed 1236.

Metric: effective causal TFLOP/s = 4 * head_dim * num_heads * (visible (query,
key) pairs) / time, with the fraction of the measured dense-bf16 tensor peak.

One "step" = one b2pa_context_attention call over the whole batch (one
attention kernel, which also sorts its work items).  Inputs are resident in HBM; L2 is flushed (a 512 MiB
write) before every timed step, outside the timed events.  Prints one JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores on a bounded row
sample of the same workload (there is no other reference implementation).
Under torchrun with N > 1 every rank runs its own replica (no collective on
the data path); value = all ranks' work / the slowest rank's time.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload  # noqa: E402

METRIC = "effective causal TFLOPS of paged prefill attention and % of GB300 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD_INDEX = 2
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_tc_llama3_8b_prefill_traffic.json")
KERNEL_SOURCES = ["attn_tc.cu", "attn_common.cuh", "common.cuh", "ptx.cuh", "worklist.cuh"]


# --------------------------------------------------------------------------- workload arithmetic

def visible_pairs(inp) -> int:
    """Sum over requests and queries of the number of visible keys (per head)."""
    total = 0
    W = inp.window_left
    for ql, kl in zip(inp.q_lens, inp.kv_lens):
        if ql <= 0:
            continue
        pos = np.arange(kl - ql, kl, dtype=np.int64)
        vis = pos + 1 if W < 0 else np.minimum(pos + 1, W + 1)
        total += int(vis.sum())
    return total


def step_flops(inp) -> float:
    return 4.0 * inp.head_dim * inp.num_heads * visible_pairs(inp)


def workload_config(inp, l2: str) -> dict:
    return {
        "workload": inp.name,
        "batch": inp.batch,
        "num_tokens": int(inp.q.shape[0]),
        "num_heads": inp.num_heads,
        "num_kv_heads": inp.num_kv_heads,
        "head_dim": inp.head_dim,
        "page_size": inp.page_size,
        "kv_layout": inp.layout,
        "kv_dtype": inp.meta.get("kv_dtype"),
        "seed": inp.seed,
        "visible_pairs_per_head": visible_pairs(inp),
        "l2": l2,
        "parallelism": "replicas",
    }


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["bf16_tflops"]), float(p.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "paged_kv_prefill_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    t = json.load(open(TRAFFIC_FILE))
    if t.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return t.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        os.unlink(self.path)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        load = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4) if r[6 + i].lower().startswith("active")})
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons,
            "samples": len(rows),
            "samples_under_load": len(load),
            "power_w_max": max((num(r[3]) or 0) for r in rows) if rows else None,
        }


# --------------------------------------------------------------------------- distributed helpers

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle timing

def oracle_rows(inp, fraction: float, seed: int) -> np.ndarray:
    T, H = inp.q.shape[0], inp.num_heads
    n = max(1, int(T * H * fraction))
    g = np.random.default_rng(seed)
    return np.sort(g.choice(T * H, size=n, replace=False)).astype(np.int64)


def rows_pairs(inp, rows: np.ndarray) -> int:
    H = inp.num_heads
    cq = inp.cum_q.numpy().astype(np.int64)
    kv = inp.seq_lens.numpy().astype(np.int64)
    tok = rows // H
    b = np.searchsorted(cq, tok, side="right") - 1
    i = tok - cq[b]
    pos = kv[b] - (cq[b + 1] - cq[b]) + i
    W = inp.window_left
    vis = pos + 1 if W < 0 else np.minimum(pos + 1, W + 1)
    return int(vis.sum())


def time_oracle(inp, rows):
    import oracle

    t0 = time.perf_counter()
    _, st, threads = oracle.attention(inp, rows=rows)
    dt = time.perf_counter() - t0
    assert (st == 0).all()
    flops = 4.0 * inp.head_dim * rows_pairs(inp, rows)
    return flops, dt, threads


# --------------------------------------------------------------------------- our arm

def run_all_workloads(reps: int = 20):
    """One JSON line per named workload (not the bench contract line): median
    device time of the attention kernel alone and of the whole call, each
    after a 512 MiB L2 flush, with effective TFLOP/s and algorithmic GB/s."""
    import paged_kv_prefill_gb300 as b2pa
    from paged_kv_prefill_gb300 import build as b2pa_build

    b2pa_build.build()
    b2pa.load()
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for idx, W in [(2, None), (3, None), (4, None), (4, -1), (5, None)]:
        inp = workload.config(idx, window_left=W)
        d = {n: getattr(inp, n).to(dev) for n in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q",
                                                  "cum_kv")}
        sinks = None if inp.sinks is None else inp.sinks.to(dev)
        out = torch.empty_like(d["q"])

        def call():
            b2pa.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                   inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"],
                                   d["cum_kv"], inp.window_left, out, inp.layout, sinks, stream=stream)

        for _ in range(5):
            call()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(reps)] for _ in range(4)]
        for e in ev[0] + ev[1]:
            e.record(stream)  # the CUDA event exists once recorded
        torch.cuda.synchronize()
        for i in range(reps):
            flush.fill_(i)
            b2pa.set_timing_events(ev[0][i], ev[1][i])
            call()
            b2pa.set_timing_events(None, None)
            flush.fill_(i + 1)
            ev[2][i].record(stream)
            call()
            ev[3][i].record(stream)
        torch.cuda.synchronize()
        k_ms = statistics.median(a.elapsed_time(b) for a, b in zip(ev[0], ev[1]))
        c_ms = statistics.median(a.elapsed_time(b) for a, b in zip(ev[2], ev[3]))
        fl, by = step_flops(inp), algorithmic_bytes(inp)
        print(json.dumps({"workload": inp.name, "path": b2pa.query_path(d["q"], (d["k_pool"], d["v_pool"]), out,
                                                                        inp.layout),
                          "gflop": fl / 1e9, "algorithmic_mb": by / 1e6, "kernel_ms": k_ms, "call_ms": c_ms,
                          "kernel_tflops": fl / k_ms / 1e9, "call_tflops": fl / c_ms / 1e9,
                          "kernel_gbs": by / k_ms / 1e6, "device_status": b2pa.device_status()}), flush=True)
    run_decode_workloads(reps)
    run_append_workloads(reps)


def run_decode_workloads(reps: int = 20):
    """One JSON line per decode batch (b2pa_batch_decode): median time of the
    whole call (attention over kv chunks, then the combine) after a 512 MiB L2
    flush, with algorithmic GB/s against the copy peak; decode streams the KV
    cache once, so HBM bandwidth is its roof."""
    import paged_kv_prefill_gb300 as b2pa
    from paged_kv_prefill_gb300 import build as b2pa_build

    b2pa_build.build()
    b2pa.load()
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    _, hbm_gbs, _ = peaks()
    for n, kvd in [(1, "bf16"), (4, "bf16"), (1, "fp8_e4m3")]:
        inp = workload.decode_config(n, kv_dtype=kvd)
        d = {k: getattr(inp, k).to(dev) for k in ("q", "k_pool", "v_pool", "block_tables", "seq_lens")}
        out = torch.empty_like(d["q"])

        def call():
            b2pa.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_kv_len,
                              inp.bmm1_scale, inp.bmm2_scale, -1, out, inp.layout, None, q_len_per_req=n,
                              stream=stream)

        for _ in range(5):
            call()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(reps)] for _ in range(2)]
        torch.cuda.synchronize()
        for i in range(reps):
            flush.fill_(i)
            ev[0][i].record(stream)
            call()
            ev[1][i].record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in zip(ev[0], ev[1]))
        by = algorithmic_bytes(inp)
        print(json.dumps({"workload": inp.name, "q_len_per_req": n, "call_ms": ms, "algorithmic_mb": by / 1e6,
                          "call_gbs": by / ms / 1e6, "frac_of_copy_peak": by / ms / 1e6 / hbm_gbs,
                          "call_tflops": step_flops(inp) / ms / 1e9, "device_status": b2pa.device_status()}),
              flush=True)


def run_append_workloads(reps: int = 20):
    """One JSON line per timed K/V write (the step before the attention): every new
    token of the bench workload (bf16 pool) and of the ragged FP8 workload (e4m3
    pool) into its slot; median device time after a 512 MiB L2 flush."""
    import paged_kv_prefill_gb300 as b2pa
    from paged_kv_prefill_gb300 import build as b2pa_build

    b2pa_build.build()
    b2pa.load()
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    _, hbm_gbs, _ = peaks()
    for idx in (2, 5):
        inp = workload.config(idx)
        T, H, D = inp.q.shape[0], inp.num_kv_heads, inp.head_dim
        g = torch.Generator().manual_seed(7)
        k_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16).to(dev)
        v_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16).to(dev)
        loc = new_token_slots(inp).to(dev)
        kp, vp = inp.k_pool.to(dev), inp.v_pool.to(dev)
        ks, vs = inp.meta["k_scale"], inp.meta["v_scale"]

        def append():
            b2pa.append_kv(k_new, v_new, (kp, vp), loc, ks, vs, inp.layout, stream=stream)

        for _ in range(5):
            append()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(reps)] for _ in range(2)]
        torch.cuda.synchronize()
        for i in range(reps):
            flush.fill_(i)
            ev[0][i].record(stream)
            append()
            ev[1][i].record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in zip(ev[0], ev[1]))
        esize = kp.element_size()
        by = 2 * T * H * D * 2 + 2 * T * H * D * esize + 4 * T  # bf16 rows in, pool rows out, slots
        print(json.dumps({"workload": f"append_kv:{inp.name}", "pool_dtype": str(kp.dtype).replace("torch.", ""),
                          "tokens": T, "algorithmic_mb": by / 1e6, "kernel_ms": ms, "kernel_gbs": by / ms / 1e6,
                          "frac_of_copy_peak": by / ms / 1e6 / hbm_gbs, "device_status": b2pa.device_status()}),
              flush=True)


def new_token_slots(inp):
    """cache_loc of each request's new tokens (positions kv_len - q_len .. kv_len - 1) through its page table."""
    P = inp.page_size
    loc = []
    for b in range(inp.batch):
        q_len = int(inp.cum_q[b + 1] - inp.cum_q[b])
        kv = int(inp.seq_lens[b])
        pos = torch.arange(kv - q_len, kv)
        loc.append(inp.block_tables[b].long()[pos // P] * P + pos % P)
    return torch.cat(loc).to(torch.int32)


def run_profile_workload(name: str, warmup: int, steps: int):
    """For ncu: W warm-up calls then K calls of another named workload (the
    sliding-window layer or a decode batch), each after an L2 flush; prints no
    measurement."""
    import paged_kv_prefill_gb300 as b2pa
    from paged_kv_prefill_gb300 import build as b2pa_build

    b2pa_build.build()
    b2pa.load()
    dev = torch.device("cuda", 0)
    decode = name == "decode_q1"
    inp = workload.decode_config(1) if decode else workload.config(4)
    d = {n: getattr(inp, n).to(dev) for n in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q", "cum_kv")}
    sinks = None if inp.sinks is None else inp.sinks.to(dev)
    out = torch.empty_like(d["q"])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    for i in range(warmup + steps):
        flush.fill_(i)
        if decode:
            b2pa.batch_decode(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"], inp.max_kv_len,
                              inp.bmm1_scale, inp.bmm2_scale, inp.window_left, out, inp.layout, sinks,
                              q_len_per_req=1)
        else:
            b2pa.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                   inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"],
                                   d["cum_kv"], inp.window_left, out, inp.layout, sinks)
    torch.cuda.synchronize()
    print(f"profile run ({inp.name}): {warmup} + {steps} calls, device bits {b2pa.device_status()}", flush=True)


def run_ours(args, world, rank, local):
    import paged_kv_prefill_gb300 as b2pa
    from paged_kv_prefill_gb300 import build as b2pa_build

    if rank == 0 or world == 1:
        b2pa_build.build()
    barrier(world)
    b2pa.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workload.config(WORKLOAD_INDEX)
    flops = step_flops(inp)
    q = inp.q.to(dev)
    k = inp.k_pool.to(dev)
    v = inp.v_pool.to(dev)
    bt = inp.block_tables.to(dev)
    sl = inp.seq_lens.to(dev)
    cq = inp.cum_q.to(dev)
    ck = inp.cum_kv.to(dev)
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(qq=q, oo=out):
        b2pa.context_attention(qq, (k, v), bt, sl, inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale,
                               cq, ck, inp.window_left, oo, inp.layout, None, stream=stream)

    assert b2pa.query_path(q, (k, v), out, inp.layout) == "tcgen05"
    if args.profile:
        # for ncu: W warm-up calls then K calls, nothing else (no numbers are reported)
        for i in range(args.warmup + args.steps):
            flush.fill_(i)
            call()
        torch.cuda.synchronize()
        print(f"profile run: {args.warmup} + {args.steps} calls, device bits {b2pa.device_status()}", flush=True)
        return
    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    sampler.start()
    # bring the clocks up (not timed), then warm up
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        for _ in range(20):
            call()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        flush.fill_(1)
        call()
    torch.cuda.synchronize()
    bits = b2pa.device_status()
    if bits:
        raise RuntimeError(f"device error bits {bits} during warm-up")

    # ---- timed region: K steps, each bracketed by events; L2 flushed outside the events
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i)
        ev0[i].record(stream)
        call()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms = sum(step_ms)
    total_ms_max = max_over_ranks(total_ms, world, dev)
    all_flops = sum_over_ranks(flops * K, world, dev)
    value = all_flops / (total_ms_max * 1e-3) / 1e12

    # ---- the attention kernel alone: events recorded by the library around its launch
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ka + kb:
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i)
        b2pa.set_timing_events(ka[i], kb[i])
        call()
    b2pa.set_timing_events(None, None)
    torch.cuda.synchronize()
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ka, kb))
    bits = b2pa.device_status()
    if bits:
        raise RuntimeError(f"device error bits {bits} during the timed region")

    # ---- end to end through the public call with host buffers: H2D inputs, call, D2H result.
    # Every step copies its own inputs from pinned host memory and reads its result
    # back; steps are pipelined on three streams (copies in, the call, copies out)
    # with two device buffers, so one step's copies overlap another's kernels.
    # E = the steps' work over the wall time from the first copy to the last read.
    host = {n: getattr(inp, n).pin_memory() for n in ("q", "k_pool", "v_pool", "block_tables", "seq_lens", "cum_q",
                                                       "cum_kv")}
    dbufs = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_hosts = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    Ke = max(3, min(K, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        done_in = [torch.cuda.Event() for _ in range(n)]
        done_call = [torch.cuda.Event() for _ in range(n)]
        done_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done_call[i - 2])  # buffer b is free once call i-2 is done
                for name in host:
                    dbufs[b][name].copy_(host[name], non_blocking=True)
                done_in[i].record(s_in)
            stream.wait_event(done_in[i])
            if i >= 2:
                stream.wait_event(done_out[i - 2])  # outs[b] has been read back
            d = dbufs[b]
            b2pa.context_attention(d["q"], (d["k_pool"], d["v_pool"]), d["block_tables"], d["seq_lens"],
                                   inp.max_q_len, inp.max_kv_len, inp.bmm1_scale, inp.bmm2_scale, d["cum_q"],
                                   d["cum_kv"], inp.window_left, outs[b], inp.layout, None, stream=stream)
            done_call[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_call[i])
                out_hosts[b].copy_(outs[b], non_blocking=True)
                done_out[i].record(s_out)
        return done_out

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    for cs in (stream, s_out):
        cs.wait_event(e_start)
    last = e2e_run(Ke)
    s_out.wait_event(last[-1])
    e_end.record(s_out)
    torch.cuda.synchronize()
    if not torch.equal(out_hosts[(Ke - 1) % 2], out.cpu()):
        raise RuntimeError("end-to-end result differs from the device-timed result")
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), world, dev)
    e2e_value = sum_over_ranks(flops * Ke, world, dev) / (e2e_ms * 1e-3) / 1e12

    peak_tf, hbm_gbs, peak_src = peaks()
    achieved = flops / (kern_ms * 1e-3) / 1e12
    traffic = recorded_traffic()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = oracle_rows(inp, args.cpu_fraction, seed=1)
        f, dt, threads = time_oracle(inp, rows)
        cpu = {"value": f / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{len(rows)} of {inp.q.shape[0] * inp.num_heads} (token, head) rows "
                         f"({args.cpu_fraction:.3f} of the batch, seeded), fp64, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": total_ms_max / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config(inp, "flushed: 512 MiB write before every timed step, outside the events"),
            "fraction_of_peak": value / peak_tf,
            "roofline": {
                "bound": "tensor",
                "achieved": achieved,
                "peak": peak_tf,
                "unit": UNIT,
                "frac": achieved / peak_tf,
                "traffic": traffic,
                "peak_source": f"{peak_src} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                if peak_src == "measured" else "fallback 1.9 PFLOP/s bf16",
                "kernel": "attention_tc_kernel<128,false>",
                "kernel_ms": kern_ms,
                "flops_per_launch": flops,
                "algorithmic_bytes_per_launch": algorithmic_bytes(inp),
                "achieved_hbm_gbs": algorithmic_bytes(inp) / (kern_ms * 1e-3) / 1e9,
                "hbm_peak_gbs": hbm_gbs,
            },
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": Ke, "pipeline": "copies in / call / copies out on three streams, two device buffers"},
            "gpu_launches": K,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)


def algorithmic_bytes(inp) -> int:
    """Bytes one launch must move at least: Q and O once, each used K/V token once per kv head."""
    T, H, D = inp.q.shape
    qo = 2 * T * H * D * 2
    kv_tok = sum(inp.kv_lens)
    es = 1 if inp.meta.get("kv_dtype") == "fp8_e4m3" else 2
    kv = 2 * kv_tok * inp.num_kv_heads * D * es
    tables = inp.block_tables.numel() * 4 + (inp.batch * 3 + 2) * 4
    return qo + kv + tables


# --------------------------------------------------------------------------- reference arm (the CPU oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    inp = workload.config(WORKLOAD_INDEX)
    # size each step so that warm-up + timed steps take about two minutes
    probe = oracle_rows(inp, 0.01, seed=2)
    f, dt, threads = time_oracle(inp, probe)
    rate = f / dt
    steps = args.steps + args.warmup
    budget = min(10.0, 120.0 / max(1, steps))
    fraction = min(1.0, budget * rate / step_flops(inp))
    for i in range(args.warmup):
        time_oracle(inp, oracle_rows(inp, fraction, seed=100 + i))
    tot_f = tot_t = 0.0
    for i in range(args.steps):
        f, dt, threads = time_oracle(inp, oracle_rows(inp, fraction, seed=1000 + i))
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    sample = (f"each step: {fraction:.4f} of the batch's (token, head) rows, seeded, fp64 CPU oracle, "
              f"{tot_t / args.steps:.2f} s per step")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(inp, "n/a (host CPU)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-fraction", type=float, default=0.125)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-workloads", action="store_true",
                    help="time every named workload (kernel and call) and the K/V writes instead of the bench line")
    ap.add_argument("--append", action="store_true",
                    help="time only the K/V writes (b2pa_append_kv) of the bench and ragged FP8 workloads")
    ap.add_argument("--decode", action="store_true",
                    help="time only the decode batches (b2pa_batch_decode)")
    ap.add_argument("--profile", action="store_true",
                    help="only W + K calls of the workload (for ncu); prints no measurement")
    ap.add_argument("--profile-workload", choices=["swa127", "decode_q1"],
                    help="as --profile, for the sliding-window layer or the q_len_per_req 1 decode batch")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.all_workloads:
        run_all_workloads()
        return
    if args.append:
        run_append_workloads()
        return
    if args.decode:
        run_decode_workloads()
        return
    if args.profile_workload:
        run_profile_workload(args.profile_workload, args.warmup, args.steps)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
