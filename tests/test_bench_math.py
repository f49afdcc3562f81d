"""The bench's arithmetic on the CPU: workload byte counts against their closed forms for the
workloads' stated shapes, the combined roofline fraction, whole-job throughput and the
counter deltas of a timed region."""
import math

import pytest

import bench
import workload as W


def test_qwen_byte_counts_closed_form():
    """Qwen3-14B-shaped decode: 32 requests of 32,768 tokens, 8 layers, 8 KV heads, 64-token
    partitions of 128-wide bf16 K and V, top-32, fp32 summaries."""
    w = W.by_name("qwen3_14b_32k")
    parts = 32768 // 64
    assert w.summary_bytes_per_step() == 32 * 8 * 8 * parts * 128 * 4 == 512 * 2**20
    assert w.selected_kv_bytes_per_step() == 32 * 8 * 8 * 32 * (2 * 64 * 128 * 2) == 2 * 2**30
    assert w.host_kv_bytes() == 32 * 8 * 8 * parts * (2 * 64 * 128 * 2) == 32 * 2**30


def test_long_request_byte_counts_closed_form():
    """One 1M-token request: 16,384 partitions per head, top-128 of them."""
    w = W.by_name("long_1m")
    assert w.summary_bytes_per_step() == 8 * 16384 * 128 * 4 == 64 * 2**20
    assert w.selected_kv_bytes_per_step() == 8 * 128 * 32768 == 32 * 2**20


def test_selected_bytes_cap_at_partitions():
    """A request with fewer partitions than k selects all of them."""
    w = W.Workload("short", B=2, L=1, Hq=2, Hkv=2, ctx_len=[64 * 3, 64 * 40], topk=8, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=0)
    assert w.selected_kv_bytes_per_step() == (3 + 8) * 2 * 32768


def test_roofline_terms_definition():
    """(selected / HBM + retrieved / link) / time, and the same plus the summaries' HBM time."""
    w = W.by_name("long_1m")
    d = {"selected_bytes": 2 * 10**9, "retrieved_bytes": 10**9}
    r = bench.roofline_terms(w, d, ms_total=1000.0, hbm_gbs=4.0, host_gbs=2.0, steps=2)
    ideal = 2e9 / 4e9 + 1e9 / 2e9
    assert math.isclose(r["frac"], ideal / 1.0)
    assert math.isclose(r["frac_with_summaries"], (ideal + 2 * w.summary_bytes_per_step() / 4e9) / 1.0)
    assert bench.roofline_terms(w, d, 0.0, 4.0, 2.0, 1) == {"frac": None, "frac_with_summaries": None}


def test_job_tokens_per_s_uses_all_ranks_over_the_slowest():
    assert math.isclose(bench.job_tokens_per_s(32 * 20, 4, 2000.0), 32 * 20 * 4 / 2.0)


def test_stats_delta_subtracts_every_counter():
    keys = ("hits", "misses", "evictions", "retrieved_bytes", "selected_bytes", "timed_calls", "ms_score",
            "ms_manage", "ms_pages", "ms_combine", "ms_kernel", "lru_rounds", "steps")
    st0 = {k: i for i, k in enumerate(keys)}
    st1 = {k: 10 * i + 7 for i, k in enumerate(keys)}
    d = bench.stats_delta(st1, st0)
    assert d == {k: 9 * i + 7 for i, k in enumerate(keys)}


@pytest.mark.parametrize("text,cpus", [("0-3", {0, 1, 2, 3}), ("0-1,8,10-11\n", {0, 1, 8, 10, 11}), ("", set())])
def test_parse_cpulist(text, cpus):
    assert bench.parse_cpulist(text) == cpus
