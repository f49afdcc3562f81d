#!/usr/bin/env python3
"""Benchmark of the SPIN sparse-decode data path on GB300.

One step = one decode step of the whole workload: every layer's call of
spin_decode_step (Select -> two-level resolve -> bucketed LRU -> Retrieve ->
sparse attention -> combine) over the whole batch. The default workload is the
Qwen3-14B-shaped batch (32 requests x 8 layers x 8 KV heads, 32K tokens,
top-32 partitions, 5x buffer). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl spin|reference]
                  [--workload NAME] [--layers L] [--batch B] [--no-e2e] [--no-cpu-baseline]

--impl reference times the CPU oracle (the plain double-precision restatement)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload as W  # noqa: E402

METRIC = "sparse decode tokens/s on 1 GB300; achieved HBM & host-link GB/s vs roofline"
PAGE_BYTES = 32768
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="spin", choices=["spin", "reference"])
    ap.add_argument("--workload", default="qwen3_14b_32k", choices=sorted(W.ALL))
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling runs)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling runs)")
    ap.add_argument("--mean-part", type=int, default=0,
                    help="variable partitions of 1-64 tokens averaging about this many (a seeded grouping)")
    ap.add_argument("--append", action="store_true",
                    help="KV append: one new token per request per layer before every decode step (tail mode)")
    ap.add_argument("--budget", type=int, default=0,
                    help="resident budget in pages per unit for every request (buffer elasticity), topk..cap")
    ap.add_argument("--tier-split", action="store_true",
                    help="second-level segment entries in pinned host memory")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU work of the oracle sample")
    ap.add_argument("--host-alloc", default="cuda", choices=["cuda", "hugepages"],
                    help="pinned host page store: cudaHostAlloc (default) or huge-page mmap + cudaHostRegister")
    return ap.parse_args()


class Ranks:
    """One process per GPU (torchrun env). Shards are independent batches: rank r runs
    the workload drawn with seed r, so per-GPU work is fixed as ranks are added
    (weak scaling). The only collectives are a barrier and max-over-ranks timing."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dev = None

    def init(self, backend: str, device=None):
        self.dev = device
        if self.world > 1:
            import torch.distributed as dist
            kw = {"device_id": device} if (backend == "nccl" and device is not None) else {}
            dist.init_process_group(backend, **kw)

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return float(x)
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.dev if self.dev is not None else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


def job_tokens_per_s(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the tokens of all ranks over the slowest rank's time."""
    return tokens_per_rank * world / (max_ms * 1e-3)


def make_workload(args, rank=0):
    w = W.by_name(args.workload, seed=rank)
    if args.layers:
        w = w.with_(L=args.layers)
    if args.batch:
        w = w.with_(B=args.batch, ctx_len=w.ctx_len[:args.batch])
    if getattr(args, "mean_part", 0):
        w = w.with_(mean_part=args.mean_part)
    return w


def workload_desc(w):
    ctx = w.ctx_len
    ctx_s = str(ctx[0]) if len(set(ctx)) == 1 else f"{min(ctx)}-{max(ctx)} (mean {int(np.mean(ctx))})"
    parts = "64-token partitions"
    if w.mean_part:
        n_p = sum(w.var_partitions(b) for b in range(w.B))
        parts = (f"variable partitions of 1-64 tokens (mean {sum(ctx) / max(n_p, 1):.1f}, "
                 f"seeded grouping within 256-token windows)")
    return (f"{w.name}: batch {w.B}, {w.L} layers, {w.Hq} q / {w.Hkv} kv heads, head_dim 128, context {ctx_s} tokens, "
            f"{parts}, top-{w.topk}, buffer {w.buf_mult}x, drift {w.drift_a}/{w.drift_c}, seed {w.seed}")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def host_link_peak_gbs(torch, dev, nbytes=1 << 30, reps=5):
    """Pinned host -> device cudaMemcpyAsync bandwidth (1 GiB copies, best of reps)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def attention_traffic(ppl_bytes):
    """Per-launch DRAM bytes of the attention kernel from the committed ncu summary, when it
    was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    src = os.path.join(ROOT, "sparse_attention_tiered_gb300", "csrc", "k_attend.cu")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    if d.get("source_sha256") != h:
        return None
    # scale the captured launch to this workload's per-launch selected bytes
    return int(d["dram_bytes_per_selected_byte"] * ppl_bytes)


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def run_oracle_sample(w, steps_budget, cpu_seconds):
    """Times the oracle on the units of request 0 (all layers, all KV heads) for as many
    decode steps as fit in about `cpu_seconds`; returns (tokens/s, threads, sample text)."""
    import oracle as O
    units, qgroup = [], []
    for l in range(w.L):
        k, v = w.request_kv(l, 0)
        order, starts = w.request_parts(l, 0) if w.mean_part else (None, None)
        for h in range(w.Hkv):
            if w.mean_part:
                units.append(O.Unit.from_parts(np.ascontiguousarray(k[h]), np.ascontiguousarray(v[h]), order[h],
                                               starts[h], w.cap))
            else:
                units.append(O.Unit(w.ctx_len[0], w.cap, np.ascontiguousarray(k[h]), np.ascontiguousarray(v[h])))
            qgroup.append((l, h))
        del k, v
    qs = w.queries()
    threads = os.cpu_count() or 1
    done, elapsed, t = 0, 0.0, 0
    while t < max(1, steps_budget):
        qb = qs.bf16()
        per_unit = [np.ascontiguousarray(qb[l, 0, h * w.G:(h + 1) * w.G]) for (l, h) in qgroup]
        t0 = time.perf_counter()
        used, _ = O.step_units_parallel(units, per_unit, w.topk, t, threads=threads)
        dt = time.perf_counter() - t0
        if t > 0:  # the first step (all misses) is the warm-up
            elapsed += dt
            done += 1
        threads = used
        qs.advance()
        t += 1
        if elapsed >= cpu_seconds:
            break
    tok_s = done / elapsed if elapsed > 0 else 0.0  # one request -> one token per decode step
    sample = (f"request 0 only ({w.L} layers x {w.Hkv} KV heads = {len(units)} units of {w.units}), "
              f"{done} timed decode steps after 1 warm-up step, {elapsed:.1f} s")
    return tok_s, threads, sample


def bench_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = make_workload(args)
    steps = args.steps
    tok_s, threads, sample = run_oracle_sample(w, 100000, args.cpu_seconds)
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 / tok_s if tok_s else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": workload_desc(w), "sample": "oracle on host cores"},
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU path
# ---------------------------------------------------------------------------

def bench_spin(args):
    import torch
    from sparse_attention_tiered_gb300 import SpinContext
    from sparse_attention_tiered_gb300._binding import (SPIN_FLAG_HOST_HUGEPAGES, SPIN_FLAG_STAGE_TIMING,
                                                        SPIN_FLAG_TIER_SPLIT)

    R = Ranks()
    world, rank, local = R.world, R.rank, R.local
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    R.init("nccl", dev)

    def barrier():
        R.barrier()
        torch.cuda.synchronize()

    w = make_workload(args, rank)
    K, Wm = args.steps, max(3, args.warmup)
    n_steps_total = Wm + K + (0 if args.no_e2e else K)
    if args.append and w.mean_part:
        raise SystemExit("--append and --mean-part cannot be combined (tail mode has fixed partitions)")
    if args.budget and not (w.topk <= args.budget <= w.cap):
        raise SystemExit(f"--budget must be in [{w.topk}, {w.cap}]")

    # ---- set-up (untimed): Index + Offload of every request and layer ----
    t_setup = time.perf_counter()
    flags = SPIN_FLAG_STAGE_TIMING | (SPIN_FLAG_HOST_HUGEPAGES if args.host_alloc == "hugepages" else 0)
    flags |= SPIN_FLAG_TIER_SPLIT if args.tier_split else 0
    ctx = SpinContext.for_workload(w, device=local, flags=flags,
                                   **({"append_tokens": n_steps_total} if args.append else {}))
    kbuf = vbuf = None
    keep = []
    for l in range(w.L):
        for b in range(w.B):
            n = w.ctx_len[b]
            if kbuf is None or kbuf.shape[1] != n:
                torch.cuda.synchronize()
                keep = [torch.empty((w.Hkv, n, 128), dtype=torch.int16).pin_memory() for _ in range(2)]
                kbuf, vbuf = (t_.numpy().view(np.uint16) for t_ in keep)
            w.request_kv(l, b, kbuf, vbuf)
            if w.mean_part:
                ctx.index_offload_parts(b, l, kbuf, vbuf, *w.request_parts(l, b))
            else:
                ctx.index_offload_host(b, l, kbuf, vbuf)
            torch.cuda.synchronize()
    if args.budget:
        for b in range(w.B):
            ctx.set_buffer(b, args.budget)
        torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    # ---- appended tokens (tail mode): seeded bf16 N(0,1) K and V, [step][layer][k|v][B][Hkv][128] ----
    kv_host = kv_dev = kv_stage = None
    if args.append:
        gen = torch.Generator().manual_seed(1000 + rank)
        kv_host = torch.randn((n_steps_total, w.L, 2, w.B, w.Hkv, 128), generator=gen).to(torch.bfloat16)
        kv_host = kv_host.view(torch.int16).pin_memory()
        kv_dev = kv_host[:Wm + K].to(dev)
        kv_stage = torch.empty((2, w.B, w.Hkv, 128), dtype=torch.int16, device=dev)

    # ---- queries for every step, resident in HBM (and pinned on the host for e2e) ----
    qs = w.queries()
    q_host = torch.empty((n_steps_total, w.L, w.B, w.Hq, 128), dtype=torch.int16).pin_memory()
    for t in range(n_steps_total):
        q_host[t].copy_(torch.from_numpy(qs.bf16().view(np.int16)))
        qs.advance()
    q_dev = q_host[:Wm + K].to(dev)
    out = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def step(t):
        for l in range(w.L):
            if args.append:
                ctx.append_kv(l, kv_dev[t, l, 0], kv_dev[t, l, 1], stream)
            ctx.decode_step(l, q_dev[t, l], out[l], stream)

    hbm_gbs, peak_src = measured_peaks()
    host_gbs = host_link_peak_gbs(torch, dev)

    for t in range(Wm):
        step(t)
    torch.cuda.synchronize()
    st0 = ctx.stats()

    # ---- timed region: K steps, inputs resident ----
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(Wm, Wm + K):
        step(t)
    e1.record()
    barrier()
    clk = clocks.stop()
    ms_rank = e0.elapsed_time(e1)
    st1 = ctx.stats()
    ms = R.max(ms_rank)
    value = job_tokens_per_s(w.B * K, world, ms)

    d = {k2: st1[k2] - st0[k2] for k2 in ("hits", "misses", "evictions", "retrieved_bytes", "selected_bytes",
                                          "timed_calls", "ms_select", "ms_manage", "ms_retrieve", "ms_attention",
                                          "ms_combine", "lru_rounds")}
    calls = max(1, d["timed_calls"])
    att_ms = d["ms_attention"] / calls          # the fused retrieve + attention kernel, per layer call
    sel_bytes_per_launch = d["selected_bytes"] / calls
    ret_bytes_per_launch = d["retrieved_bytes"] / calls
    hbm_achieved = sel_bytes_per_launch / (att_ms * 1e-3) / 1e9 if att_ms > 0 else 0.0
    host_achieved = ret_bytes_per_launch / (att_ms * 1e-3) / 1e9 if att_ms > 0 else 0.0
    host_bound = ret_bytes_per_launch / host_gbs >= sel_bytes_per_launch / hbm_gbs
    traffic = attention_traffic(sel_bytes_per_launch)
    combined_ideal_s = d["selected_bytes"] / (hbm_gbs * 1e9) + d["retrieved_bytes"] / (host_gbs * 1e9)
    summ_ideal_s = K * w.summary_bytes_per_step() / (hbm_gbs * 1e9)
    gpu_launches = K * w.L * ((2 if (w.B * w.Hkv >= 64 and w.p_max <= 4096) else 3) + (1 if args.append else 0))

    # ---- end to end through the host-buffer entry point ----
    e2e = None
    if not args.no_e2e:
        o_host = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32).pin_memory()
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for t in range(Wm + K, Wm + 2 * K):
            for l in range(w.L):
                if args.append:  # the new token's K and V come from host memory too
                    kv_stage.copy_(kv_host[t, l], non_blocking=True)
                    ctx.append_kv(l, kv_stage[0], kv_stage[1], stream)
                ctx.decode_step_host(l, q_host[t, l].data_ptr(), o_host[l].data_ptr(), stream)
        a1.record()
        barrier()
        ms_e2e = R.max(a0.elapsed_time(a1))
        e2e = {"value": job_tokens_per_s(w.B * K, world, ms_e2e), "unit": "tokens/s",
               "h2d_bytes_per_step": int(q_host[0].numel() * 2 + (kv_host[0].numel() * 2 if args.append else 0)),
               "d2h_bytes_per_step": int(o_host.numel() * 4)}
    st2 = ctx.stats()
    ctx.close()

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok_s, threads, sample = run_oracle_sample(w, 100000, args.cpu_seconds)
        cpu_base = {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, fp32 accumulate/out", "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": workload_desc(w), "l2": "inputs larger than L2 (selected KV per layer "
                       f"{w.selected_kv_bytes_per_step() // w.L / 2**20:.0f} MiB > 129 MB)",
                       "parallelism": f"dp{world} (independent requests per GPU)", "timed_decode_steps": K,
                       "first_timed_step": Wm,
                       "host_store": ("cudaHostAlloc" if args.host_alloc == "cuda"
                                      else "huge-page mmap + cudaHostRegister"),
                       **({"append": "one token per request per layer before each decode step (tail mode)"}
                          if args.append else {}),
                       **({"budget_pages_per_unit": args.budget} if args.budget else {}),
                       **({"metadata": "segment entries in pinned host memory"} if args.tier_split else {})},
            "roofline": {"bound": "host_link" if host_bound else "hbm", "kernel": "attend_retrieve_kernel",
                         "achieved": host_achieved if host_bound else hbm_achieved,
                         "peak": host_gbs if host_bound else hbm_gbs, "unit": "GB/s",
                         "frac": (host_achieved / host_gbs) if host_bound else (hbm_achieved / hbm_gbs),
                         "traffic": traffic,
                         "peak_source": ("pinned H2D cudaMemcpyAsync peak measured in this run (1 GiB)" if host_bound
                                         else (f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                                               else "fallback 6800 GB/s")),
                         "algorithmic_bytes_per_launch": {"hbm_selected_kv": sel_bytes_per_launch,
                                                          "host_retrieved": ret_bytes_per_launch},
                         "hbm": {"achieved": hbm_achieved, "peak": hbm_gbs, "frac": hbm_achieved / hbm_gbs},
                         "host_link": {"achieved": host_achieved, "peak": host_gbs, "frac": host_achieved / host_gbs},
                         "avg_launch_ms": att_ms},
            "combined_roofline": {"frac": combined_ideal_s / (ms * 1e-3) if ms else None,
                                  "frac_with_summaries": (combined_ideal_s + summ_ideal_s) / (ms * 1e-3),
                                  "hbm_gbs": hbm_gbs, "host_link_gbs": host_gbs,
                                  "selected_bytes": d["selected_bytes"], "retrieved_bytes": d["retrieved_bytes"],
                                  "definition": "(selected KV bytes / HBM GB/s + retrieved bytes / pinned H2D GB/s) "
                                                "/ measured time, over the timed steps"},
            "stages_ms_per_layer_call": {k2[3:]: d[k2] / calls for k2 in
                                         ("ms_select", "ms_manage", "ms_retrieve", "ms_attention", "ms_combine")},
            "paging": {"hits": d["hits"], "misses": d["misses"], "evictions": d["evictions"],
                       "lru_rounds": d["lru_rounds"], "live_segments": st2["live_segments"],
                       "pool_segments": st2["pool_segments"], "metadata_bytes": st2["metadata_bytes"],
                       "flat_table_bytes": st2["flat_table_bytes"]},
            "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clk, "cpu_baseline": cpu_base,
            "setup_s": setup_s,
        }
        print(json.dumps(line), flush=True)
    R.close()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return bench_reference(args)
    return bench_spin(args)


if __name__ == "__main__":
    sys.exit(main())
