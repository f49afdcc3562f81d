#!/usr/bin/env python3
"""Benchmark of the SPIN sparse-decode data path on GB300.

One step = one decode step of the whole workload: every layer's call of
spin_decode_step (Select -> two-level resolve -> bucketed LRU -> Retrieve ->
sparse attention -> combine) over the whole batch. The headline workload is the
Qwen3-14B-shaped batch (32 requests x 8 layers x 8 KV heads, 32K tokens,
top-32 partitions, 5x buffer): W warm-up steps, then K timed steps, then K steps
end to end through the host-buffer entry point. Prints one JSON line.

The line's "configs" object then records every workload (Qwen3-14B, Llama-3.1-70B,
the eviction/metadata stress at 1x and 5x buffer, the 1M-token request, tiny) over
all its configured decode steps, each on a fresh context, next to the oracle timed on
a bounded sample of the same workload, plus the Qwen workload with KV append, a 2x
resident budget and tier-split metadata.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl spin|reference]
                  [--workload NAME] [--layers L] [--batch B] [--no-e2e] [--no-cpu-baseline]
                  [--no-configs]

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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload record (every workload over all its decode steps)")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0,
                    help="target CPU work of each workload's oracle sample in the per-workload record")
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

    def sum(self, x: float) -> float:
        if self.world == 1:
            return float(x)
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.dev if self.dev is not None else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    def min(self, x: float) -> float:
        return -self.max(-x)

    def check_host_memory(self, need_bytes: int, avail_bytes=None, headroom: float = 0.9):
        """Every rank of the node pins its own host page store: the ranks' stores together
        must fit in the node's available memory (MemAvailable, less a margin). The decision
        is the same on every rank; when it fails every rank exits with the figures."""
        avail = float(avail_bytes if avail_bytes is not None else mem_available_bytes())
        need_total = self.sum(need_bytes)
        avail = self.min(avail)
        if need_total > headroom * avail:
            raise SystemExit(f"host memory: {self.world} rank(s) would pin {need_total / 2**30:.1f} GiB of page stores "
                             f"but the node has {avail / 2**30:.1f} GiB available ({headroom:.0%} usable); "
                             f"use fewer GPUs per node or a smaller workload")
        return need_total, avail

    def close(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


def mem_available_bytes(meminfo: str = "/proc/meminfo") -> int:
    """MemAvailable of the host in bytes (0 when unknown)."""
    try:
        with open(meminfo) as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def parse_cpulist(text: str):
    """CPUs of a sysfs cpulist ("0-15,32-47")."""
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def gpu_local_cpus(pci_bus_id: str, sysfs: str = "/sys"):
    """CPUs local to a GPU (its PCI device's local_cpulist), or None when unknown."""
    try:
        with open(os.path.join(sysfs, "bus", "pci", "devices", pci_bus_id.lower(), "local_cpulist")) as f:
            cpus = parse_cpulist(f.read())
        return cpus or None
    except (OSError, ValueError):
        return None


def bind_near_gpu(dev_index: int):
    """Keeps this rank's threads on the CPUs local to its GPU, so the pinned host page store,
    first touched by the allocating thread, lands in that CPU's memory (one NUMA node per
    Grace). Returns the CPUs, or None when the topology is not exposed."""
    import torch
    props = torch.cuda.get_device_properties(dev_index)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", 0)
    dv = getattr(props, "pci_device_id", None)
    if bus is None or dv is None:
        return None
    cpus = gpu_local_cpus(f"{dom:08x}:{bus:02x}:{dv:02x}.0")
    if cpus:
        try:
            os.sched_setaffinity(0, cpus & os.sched_getaffinity(0) or cpus)
        except OSError:
            return None
    return cpus


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


def host_link_peaks(torch, dev):
    """Host -> device link ceilings measured in this run (GB/s = 1e9 bytes/s), each the
    best of a few repetitions:
      copy_1x1GiB     one 1 GiB pinned -> HBM cudaMemcpyAsync
      copy_2x256MiB   two concurrent 256 MiB copies on separate streams
      copy_4x256MiB   four concurrent 256 MiB copies on separate streams
      sm_read_4GiB    SM zero-copy 16-byte reads streaming 4 GiB of pinned memory
                      (spin_measure_host_read, the retrievers' access path)
    The peak used for the roofline is the largest of them."""
    from sparse_attention_tiered_gb300 import spin_measure_host_read
    GiB = 1 << 30
    src = torch.empty(4 * GiB, dtype=torch.uint8).pin_memory()
    src[::4096] = 1
    dst = torch.empty(GiB, dtype=torch.uint8, device=dev)

    def copies(n_streams, nbytes):
        streams = [torch.cuda.Stream() for _ in range(n_streams)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        done = []
        for i, st in enumerate(streams):
            st.wait_event(a)
            with torch.cuda.stream(st):
                dst[i * nbytes:(i + 1) * nbytes].copy_(src[i * nbytes:(i + 1) * nbytes], non_blocking=True)
            e = torch.cuda.Event()
            e.record(st)
            done.append(e)
        for e in done:
            torch.cuda.current_stream().wait_event(e)
        b.record()
        torch.cuda.synchronize()
        return n_streams * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

    out = {"copy_1x1GiB": max(copies(1, GiB) for _ in range(4)),
           "copy_2x256MiB": max(copies(2, 256 << 20) for _ in range(4)),
           "copy_4x256MiB": max(copies(4, 256 << 20) for _ in range(4)),
           "sm_read_4GiB": max(spin_measure_host_read(src.data_ptr(), 4 * GiB, 1) for _ in range(3))}
    del src, dst
    torch.cuda.synchronize()
    return {k: round(v, 2) for k, v in out.items()}


def attention_traffic(ppl_bytes):
    """Per-launch DRAM bytes of the decode-step kernel from the committed ncu summary, when it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_step_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for name in ("k_step.cu", "select_dev.cuh"):
        with open(os.path.join(ROOT, "sparse_attention_tiered_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if d.get("source_sha256") != h.hexdigest():
        return None
    # scale the captured launch to this workload's per-launch algorithmic HBM bytes
    return int(d["dram_bytes_per_algorithmic_byte"] * ppl_bytes)


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def run_oracle_sample(w, steps_budget, cpu_seconds, threads=0):
    """Times the oracle on the units of request 0 (all layers, all KV heads) for as many
    decode steps as fit in about `cpu_seconds` (threads: 0 = every host core); returns
    (tokens/s, threads used, sample text)."""
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
    threads = threads or os.cpu_count() or 1
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
            "config": headline_config(w, args, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU path
# ---------------------------------------------------------------------------

def make_context(w, args, local, extra_flags=0, append_tokens=0, rank=0, stage_timing=False):
    """Context with every request of every layer indexed and offloaded (set-up, untimed).
    stage_timing: CUDA events around every launch and in-kernel stage stamps. They add a few
    microseconds to each launch, so throughput is timed on contexts without them and the
    per-launch durations and stages come from a separate pass over the same steps."""
    import torch
    from sparse_attention_tiered_gb300 import SpinContext
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_HOST_HUGEPAGES, SPIN_FLAG_STAGE_TIMING
    flags = ((SPIN_FLAG_STAGE_TIMING if stage_timing else 0) |
             (SPIN_FLAG_HOST_HUGEPAGES if args.host_alloc == "hugepages" else 0) | extra_flags)
    ctx = SpinContext.for_workload(w, device=local, flags=flags,
                                   **({"append_tokens": append_tokens} if append_tokens else {}))
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
    return ctx


def stats_delta(st1, st0):
    keys = ("hits", "misses", "evictions", "retrieved_bytes", "selected_bytes", "timed_calls", "ms_score", "ms_manage",
            "ms_pages", "ms_combine", "ms_kernel", "lru_rounds", "steps")
    return {k2: st1[k2] - st0[k2] for k2 in keys}


def roofline_terms(w, d, ms_total, hbm_gbs, host_gbs, steps):
    """Combined roofline of `steps` decode steps measured in ms_total milliseconds:
    (selected KV bytes / HBM GB/s + retrieved bytes / host-link GB/s) / measured time; the
    stricter fraction also counts the summaries Select reads."""
    ideal = d["selected_bytes"] / (hbm_gbs * 1e9) + d["retrieved_bytes"] / (host_gbs * 1e9)
    summ = steps * w.summary_bytes_per_step() / (hbm_gbs * 1e9)
    t = ms_total * 1e-3
    return {"frac": ideal / t if t else None, "frac_with_summaries": (ideal + summ) / t if t else None}


def run_config(w, args, local, hbm_gbs, host_gbs, extra_flags=0, budget=0, append=False, oracle_seconds=0.0,
               warm_steps=0):
    """Runs every decode step of a workload (its configured count) on a fresh context and
    reports throughput over all steps and over the steps after `warm_steps`, the paging
    record, the roofline fractions and, optionally, the oracle on a bounded sample. A second
    fresh context runs the same steps with stage timing for the per-launch stage record."""
    import torch
    dev = torch.device(f"cuda:{local}")
    steps = w.steps
    qs = w.queries()
    q_dev = torch.empty((steps, w.L, w.B, w.Hq, 128), dtype=torch.int16)
    for t in range(steps):
        q_dev[t].copy_(torch.from_numpy(qs.bf16().view(np.int16)))
        qs.advance()
    q_dev = q_dev.to(dev)
    kv = None
    if append:
        gen = torch.Generator().manual_seed(1000)
        kv = torch.randn((steps, w.L, 2, w.B, w.Hkv, 128), generator=gen).to(torch.bfloat16).view(torch.int16).to(dev)
    out = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def one_pass(stage_timing):
        t_setup = time.perf_counter()
        ctx = make_context(w, args, local, extra_flags, append_tokens=steps if append else 0,
                           stage_timing=stage_timing)
        if budget:
            for b in range(w.B):
                ctx.set_buffer(b, budget)
        setup_s = time.perf_counter() - t_setup
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        torch.cuda.synchronize()
        st0 = ctx.stats()
        ev[0].record()
        stw = None
        for t in range(steps):
            for l in range(w.L):
                if append:
                    ctx.append_kv(l, kv[t, l, 0], kv[t, l, 1], stream)
                ctx.decode_step(l, q_dev[t, l], out[l], stream)
            ev[t + 1].record()
            if t + 1 == warm_steps:
                torch.cuda.synchronize()
                stw = ctx.stats()
        torch.cuda.synchronize()
        st1 = ctx.stats()
        ctx.close()
        ms_step = [ev[t].elapsed_time(ev[t + 1]) for t in range(steps)]
        return setup_s, ms_step, st0, stw, st1

    setup_s, ms_step, st0, stw, st1 = one_pass(False)
    d_all = stats_delta(st1, st0)
    d_w = stats_delta(st1, stw) if stw is not None else d_all
    ms_all, ms_w = sum(ms_step), sum(ms_step[warm_steps:])
    _, _, sst0, sstw, sst1 = one_pass(True)
    ds = stats_delta(sst1, sstw if sstw is not None else sst0)
    calls_s = max(1, ds["timed_calls"])
    r = {
        "workload": workload_desc(w), "steps": steps, "steady_from_step": warm_steps,
        "tokens_per_s_all_steps": w.B * steps / (ms_all * 1e-3),
        "tokens_per_s_steady": w.B * (steps - warm_steps) / (ms_w * 1e-3) if ms_w else None,
        "ms_per_step_first": ms_step[0], "ms_per_step_steady": ms_w / max(1, steps - warm_steps),
        "combined_roofline_all_steps": roofline_terms(w, d_all, ms_all, hbm_gbs, host_gbs, steps),
        "combined_roofline_steady": roofline_terms(w, d_w, ms_w, hbm_gbs, host_gbs, steps - warm_steps),
        "host_link_gbs_steady": d_w["retrieved_bytes"] / (ms_w * 1e-3) / 1e9 if ms_w else None,
        "hbm_selected_gbs_steady": d_w["selected_bytes"] / (ms_w * 1e-3) / 1e9 if ms_w else None,
        "stages_ms_per_layer_call_steady": {k2[3:]: ds[k2] / calls_s for k2 in
                                            ("ms_score", "ms_manage", "ms_pages", "ms_combine", "ms_kernel")},
        "stages_from": "a second fresh context over the same steps with stage timing (events per launch)",
        "paging_all_steps": {"hits": d_all["hits"], "misses": d_all["misses"], "evictions": d_all["evictions"],
                             "lru_rounds": d_all["lru_rounds"], "retrieved_bytes": d_all["retrieved_bytes"]},
        "metadata": {"metadata_bytes": st1["metadata_bytes"], "flat_table_bytes": st1["flat_table_bytes"],
                     "flat_over_metadata": st1["flat_table_bytes"] / max(1, st1["metadata_bytes"]),
                     "live_segments": st1["live_segments"], "pool_segments": st1["pool_segments"]},
        "setup_s": setup_s, "device_error": st1["device_error"] or sst1["device_error"],
    }
    del q_dev, out, kv
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if oracle_seconds > 0:
        tok_s, threads, sample = run_oracle_sample(w, 100000, oracle_seconds)
        r["oracle"] = {"tokens_per_s": tok_s, "cores": threads, "sample": sample}
    return r


def headline_config(w, args, world):
    return {"workload": workload_desc(w), "l2": "inputs larger than L2 (selected KV per layer "
            f"{w.selected_kv_bytes_per_step() // w.L / 2**20:.0f} MiB > 129 MB)",
            "parallelism": f"dp{world} (independent requests per GPU)", "timed_decode_steps": args.steps,
            "first_timed_step": max(3, args.warmup),
            "host_store": "cudaHostAlloc" if args.host_alloc == "cuda" else "huge-page mmap + cudaHostRegister",
            **({"append": "one token per request per layer before each decode step (tail mode)"} if args.append else {}),
            **({"budget_pages_per_unit": args.budget} if args.budget else {}),
            **({"metadata": "segment entries in pinned host memory"} if args.tier_split else {})}


def bench_spin(args):
    import torch
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_TIER_SPLIT

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
    n_steps_total = Wm + K
    if world > 1:
        bind_near_gpu(local)
    # every rank pins its own page store (plus the step queries): they must fit together
    R.check_host_memory(w.host_kv_bytes() + n_steps_total * w.L * w.B * w.Hq * 128 * 2)
    if args.append and w.mean_part:
        raise SystemExit("--append and --mean-part cannot be combined (tail mode has fixed partitions)")
    if args.budget and not (w.topk <= args.budget <= w.cap):
        raise SystemExit(f"--budget must be in [{w.topk}, {w.cap}]")

    hbm_gbs, peak_src = measured_peaks()

    # ---- set-up (untimed): Index + Offload of every request and layer ----
    t_setup = time.perf_counter()
    ctx = make_context(w, args, local, SPIN_FLAG_TIER_SPLIT if args.tier_split else 0,
                       append_tokens=n_steps_total if args.append else 0, rank=rank)
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
        kv_dev = kv_host.to(dev)
        kv_stage = torch.empty((2, w.B, w.Hkv, 128), dtype=torch.int16, device=dev)

    # ---- queries for every step, resident in HBM (and pinned on the host for e2e) ----
    qs = w.queries()
    q_host = torch.empty((n_steps_total, w.L, w.B, w.Hq, 128), dtype=torch.int16).pin_memory()
    for t in range(n_steps_total):
        q_host[t].copy_(torch.from_numpy(qs.bf16().view(np.int16)))
        qs.advance()
    q_dev = q_host.to(dev)
    out = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def step(t):
        for l in range(w.L):
            if args.append:
                ctx.append_kv(l, kv_dev[t, l, 0], kv_dev[t, l, 1], stream)
            ctx.decode_step(l, q_dev[t, l], out[l], stream)

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

    d = stats_delta(st1, st0)
    gpu_launches = K * w.L * (1 + (1 if args.append else 0))

    st2 = ctx.stats()
    ctx.close()

    def fresh_context(stage_timing):
        c = make_context(w, args, local, SPIN_FLAG_TIER_SPLIT if args.tier_split else 0,
                         append_tokens=n_steps_total if args.append else 0, rank=rank, stage_timing=stage_timing)
        if args.budget:
            for b in range(w.B):
                c.set_buffer(b, args.budget)
        return c

    # ---- per-launch durations and stages: the same warm-up and timed steps on a fresh context
    # with stage timing (CUDA events around every launch on its stream, in-kernel stage stamps),
    # which would add a few microseconds to every launch of the timed region above ----
    ctx = fresh_context(True)
    for t in range(Wm):
        step(t)
    torch.cuda.synchronize()
    ss0 = ctx.stats()
    for t in range(Wm, Wm + K):
        step(t)
    torch.cuda.synchronize()
    ss1 = ctx.stats()
    ctx.close()
    ds = stats_delta(ss1, ss0)
    # the host-link ceilings, measured after the timed steps: pinning and freeing their 4 GiB
    # buffer just before the store's context was created has been seen to slow that context
    links = host_link_peaks(torch, dev)
    host_gbs = max(links.values())
    calls = max(1, ds["timed_calls"])
    kern_ms = ds["ms_kernel"] / calls                   # the decode-step kernel, per layer call
    sel_b = ds["selected_bytes"] / calls                # algorithmic bytes per launch
    summ_b = w.summary_bytes_per_step() / w.L
    ret_b = ds["retrieved_bytes"] / calls
    hbm_b = sel_b + summ_b
    hbm_achieved = hbm_b / (kern_ms * 1e-3) / 1e9 if kern_ms > 0 else 0.0
    host_achieved = ret_b / (kern_ms * 1e-3) / 1e9 if kern_ms > 0 else 0.0
    host_bound = ret_b / host_gbs >= hbm_b / hbm_gbs
    traffic = attention_traffic(hbm_b)
    # ---- end to end through the host-buffer entry point: a fresh context, the same warm-up
    # and the same timed step range, with q read from and out written to pinned host memory ----
    e2e = None
    if not args.no_e2e:
        ctx = fresh_context(False)
        for t in range(Wm):
            step(t)
        o_host = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32).pin_memory()
        # A serving loop reuses its pinned input and output buffers, so the GPU's translations
        # of their host pages are warm; here every step reads a new slice of q_host, so one SM
        # read pass over both buffers (untimed) stands in for that reuse.
        from sparse_attention_tiered_gb300 import spin_measure_host_read
        spin_measure_host_read(q_host.data_ptr(), q_host.numel() * 2, 1)
        spin_measure_host_read(o_host.data_ptr(), o_host.numel() * 4, 1)
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for t in range(Wm, Wm + K):
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
               "d2h_bytes_per_step": int(o_host.numel() * 4),
               "timed_steps": f"{Wm}..{Wm + K - 1} on a fresh context after the same {Wm} warm-up steps",
               "host_buffers": "pinned q (a slice per step) and out, read and written by the kernel in place; "
                               "their pages' GPU address translations warmed by one untimed SM read pass"}
        ctx.close()
    del q_dev, q_host, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok_s, threads, sample = run_oracle_sample(w, 100000, args.cpu_seconds)
        cpu_base = {"value": tok_s, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample}

    # ---- every workload, and the bench workload's variants, over all their decode steps ----
    configs = None
    if world == 1 and not args.no_configs and not (args.append or args.budget or args.tier_split or args.mean_part):
        configs = {}
        ocs = 0.0 if args.no_cpu_baseline else args.config_cpu_seconds
        for name in ("qwen3_14b_32k", "llama31_70b_128k", "stress_m1", "stress_m5", "long_1m", "tiny"):
            wc = W.by_name(name, seed=rank)
            configs[name] = run_config(wc, args, local, hbm_gbs, host_gbs, oracle_seconds=ocs, warm_steps=3)
        wq = W.by_name("qwen3_14b_32k", seed=rank)
        configs["qwen3_14b_32k+append"] = run_config(wq, args, local, hbm_gbs, host_gbs, append=True, warm_steps=3)
        configs["qwen3_14b_32k+budget_2x"] = run_config(wq, args, local, hbm_gbs, host_gbs, budget=2 * wq.topk,
                                                        warm_steps=3)
        configs["qwen3_14b_32k+tier_split"] = run_config(wq, args, local, hbm_gbs, host_gbs,
                                                         extra_flags=SPIN_FLAG_TIER_SPLIT, warm_steps=3)
        if not args.no_cpu_baseline:
            tok1, th1, sample1 = run_oracle_sample(W.tiny(rank), 100000, 3.0, threads=1)
            configs["tiny"]["oracle_1_thread"] = {"tokens_per_s": tok1, "cores": th1, "sample": sample1}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, fp32 accumulate/out", "data": "synthetic (seeded generator; no dataset)",
            "config": headline_config(w, args, world),
            "roofline": {"bound": "host_link" if host_bound else "hbm", "kernel": "decode_step_kernel",
                         "achieved": host_achieved if host_bound else hbm_achieved,
                         "peak": host_gbs if host_bound else hbm_gbs, "unit": "GB/s",
                         "frac": (host_achieved / host_gbs) if host_bound else (hbm_achieved / hbm_gbs),
                         "traffic": traffic,
                         "peak_source": ("largest host-link rate measured in this run (host_link_peaks_gbs)"
                                         if host_bound else
                                         (f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                                          else "fallback 6800 GB/s")),
                         "algorithmic_bytes_per_launch": {"hbm_selected_kv": sel_b, "hbm_summaries": summ_b,
                                                          "host_retrieved": ret_b},
                         "hbm": {"achieved": hbm_achieved, "peak": hbm_gbs, "frac": hbm_achieved / hbm_gbs},
                         "host_link": {"achieved": host_achieved, "peak": host_gbs,
                                       "frac": host_achieved / host_gbs},
                         "avg_launch_ms": kern_ms,
                         "scope": "one launch is a whole layer step (scoring, top-k and page management, "
                                  "retrieval, attention, combine); the host link idles while the first units "
                                  "are scored and managed and after the last retrieved page lands"},
            "host_link_peaks_gbs": links,
            "combined_roofline": {**roofline_terms(w, d, ms, hbm_gbs, host_gbs, K),
                                  "hbm_gbs": hbm_gbs, "host_link_gbs": host_gbs,
                                  "selected_bytes": d["selected_bytes"], "retrieved_bytes": d["retrieved_bytes"],
                                  "definition": "(selected KV bytes / HBM GB/s + retrieved bytes / host-link GB/s) "
                                                "/ measured time, over the timed steps; frac_with_summaries also "
                                                "counts the summary bytes Select reads"},
            "stages_ms_per_layer_call": {k2[3:]: ds[k2] / calls for k2 in
                                         ("ms_score", "ms_manage", "ms_pages", "ms_combine", "ms_kernel")},
            "stages_from": "the same warm-up and timed steps on a second fresh context with stage timing",
            "paging": {"hits": d["hits"], "misses": d["misses"], "evictions": d["evictions"],
                       "lru_rounds": d["lru_rounds"], "live_segments": st2["live_segments"],
                       "pool_segments": st2["pool_segments"], "metadata_bytes": st2["metadata_bytes"],
                       "flat_table_bytes": st2["flat_table_bytes"]},
            "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clk, "cpu_baseline": cpu_base,
            "setup_s": setup_s, "configs": configs,
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
