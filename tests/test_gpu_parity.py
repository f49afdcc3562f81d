"""GPU path (through the C ABI) against the oracle, element by element.

Bars: selected-partition sets and page state bit-exact (outside the 1e-5
relative tie band of the oracle's scores), outputs within max-abs 2e-3.
"""
import numpy as np
import pytest

import oracle as O
import workload as W
from parity import OUT_TOL, AllUnits, Lockstep, sample_units

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run(w, units=None, steps=None, **kw):
    ls = Lockstep(w, units=units, **kw)
    try:
        for _ in range(steps if steps is not None else w.steps):
            ls.step()
        st = ls.ctx.stats()
        assert st["device_error"] == 0
        return ls.report, st
    finally:
        ls.close()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_lockstep(seed):
    rep, st = _run(W.tiny(seed))
    assert rep.compared_units == 4 * 16
    assert rep.max_out_err <= OUT_TOL
    assert st["misses"] > 0 and st["hits"] > 0


def test_mixed_shapes_ragged_gqa5():
    """GQA 5, two layers, ragged last partitions, context shorter than a segment, evictions (2x buffer)."""
    w = W.Workload("mixed", B=3, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 130], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=24, seed=5)
    rep, st = _run(w)
    assert rep.evictions > 0 and st["evictions"] > 0
    assert rep.max_out_err <= OUT_TOL


def test_gqa8_no_buffering():
    """GQA 8 with capacity = k (1x): every changed partition evicts."""
    w = W.Workload("gqa8", B=2, L=1, Hq=16, Hkv=2, ctx_len=[8192, 3000], topk=16, buf_mult=1,
                   drift_a=0.7, drift_c=0.3, steps=20, seed=7)
    rep, st = _run(w)
    assert st["evictions"] > 0 and rep.evictions > 0


def test_empty_short_and_k_above_partitions():
    """An empty request (zero output), one-partition and few-partition requests (k > P)."""
    w = W.Workload("edge", B=4, L=1, Hq=8, Hkv=2, ctx_len=[0, 64, 200, 5000], topk=8, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=10, seed=9)
    rep, st = _run(w)
    assert rep.max_out_err <= OUT_TOL


def test_many_segments_long_unit():
    """A unit with 40 directory entries and a large top-k (P = 2560, k = 96, 3x buffer)."""
    w = W.Workload("wide", B=1, L=1, Hq=8, Hkv=1, ctx_len=[2560 * 64], topk=96, buf_mult=3,
                   drift_a=0.8, drift_c=0.2, steps=12, seed=13)
    rep, st = _run(w)
    assert st["live_segments"] > 1


def test_summaries_match_oracle_index():
    w = W.Workload("summ", B=2, L=2, Hq=4, Hkv=2, ctx_len=[777, 4096], topk=4, buf_mult=1,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=3)
    from sparse_attention_tiered_gb300 import SpinContext
    with SpinContext.for_workload(w) as ctx:
        kv = {}
        for l in range(w.L):
            for b in range(w.B):
                kv[(l, b)] = w.request_kv(l, b)
                ctx.index_offload_host(b, l, *kv[(l, b)])
        torch.cuda.synchronize()
        for (l, b), (k, v) in kv.items():
            for h in range(w.Hkv):
                got = ctx.summaries(l, b, h).astype(np.float64)
                ref = O.index(k[h])
                # fp32 sum of bf16 values then one division: within a few fp32 ulps of the exact mean
                assert np.allclose(got, ref, rtol=4e-7, atol=1e-7), np.abs(got - ref).max()


def test_device_offload_equals_host_offload():
    w = W.Workload("devoff", B=2, L=1, Hq=8, Hkv=2, ctx_len=[3000, 640], topk=4, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=4, seed=17)
    from sparse_attention_tiered_gb300 import SpinContext
    outs = []
    summs = []
    for from_dev in (False, True):
        ls = Lockstep(w, offload_from_device=from_dev)
        try:
            for _ in range(w.steps):
                ls.step(check=True)
            outs.append(ls.out.cpu().numpy())
            summs.append([ls.ctx.summaries(0, b, h) for b in range(w.B) for h in range(w.Hkv)])
        finally:
            ls.close()
    assert np.array_equal(outs[0], outs[1])
    for a, b in zip(*summs):
        assert np.array_equal(a, b)


def test_resident_pages_byte_exact():
    """Retrieve: every resident HBM page equals the oracle's host page byte for byte."""
    w = W.Workload("bytes", B=1, L=1, Hq=4, Hkv=2, ctx_len=[64 * 50 + 9], topk=6, buf_mult=2,
                   drift_a=0.7, drift_c=0.3, steps=6, seed=19)
    ls = Lockstep(w)
    try:
        for _ in range(w.steps):
            ls.step()
        ex = ls.ctx.export(0)
        for h in range(w.Hkv):
            u = ls.oracle[(0, 0, h)]
            for s, p in enumerate(ex["slot_part"][h]):
                if p < 0:
                    continue
                page = ls.ctx.read_page(0, 0, h, s)
                assert np.array_equal(page, u.host_pages[p]), f"slot {s} (partition {p}) differs"
    finally:
        ls.close()


@pytest.mark.parametrize("variant", ["pipelined", "phased", "phased_g16"])
def test_host_buffer_entry_point_matches_device(variant):
    """spin_decode_step_host gives the device entry point's bytes whether its buffers are
    mapped pinned memory (the kernel copies q into HBM at its start and writes out in
    place), pageable memory, or pinned memory at an offset that is not 16-byte aligned
    (both copied through HBM); in both kernel variants and with two 8-head tiles."""
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_PHASED
    hq = 32 if variant == "phased_g16" else 10
    w = W.Workload("hostep", B=2, L=2, Hq=hq, Hkv=2, ctx_len=[2048, 1500], topk=6, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=5, seed=23)
    flags = SPIN_FLAG_PHASED if variant == "phased" else 0
    from sparse_attention_tiered_gb300 import SpinContext
    n = w.B * w.Hq * 128
    results = {}
    for mode in ("device", "pinned", "pageable", "pinned_unaligned"):
        with SpinContext.for_workload(w, flags=flags) as ctx:
            for l in range(w.L):
                for b in range(w.B):
                    k, v = w.request_kv(l, b)
                    ctx.index_offload_host(b, l, k, v)
                    torch.cuda.synchronize()
            qs = w.queries()
            outs = []
            if mode == "pinned":
                q_buf = torch.empty(n, dtype=torch.int16).pin_memory()
                o_buf = torch.empty(n, dtype=torch.float32).pin_memory()
            elif mode == "pinned_unaligned":  # 2- and 4-byte offsets into pinned allocations
                q_buf = torch.empty(n + 8, dtype=torch.int16).pin_memory()[1:1 + n]
                o_buf = torch.empty(n + 4, dtype=torch.float32).pin_memory()[1:1 + n]
            else:
                q_buf = torch.from_numpy(np.empty(n, np.int16))
                o_buf = torch.from_numpy(np.empty(n, np.float32))
            od = torch.empty((w.B, w.Hq, 128), dtype=torch.float32, device="cuda")
            for t in range(w.steps):
                qb = qs.bf16()
                for l in range(w.L):
                    if mode == "device":
                        qd = torch.from_numpy(qb[l].view(np.int16)).cuda()
                        ctx.decode_step(l, qd, od)
                        torch.cuda.synchronize()
                        outs.append(od.cpu().numpy().reshape(-1))
                    else:
                        q_buf.copy_(torch.from_numpy(qb[l].view(np.int16).reshape(-1)))
                        o_buf.fill_(float("nan"))
                        ctx.decode_step_host(l, q_buf.data_ptr(), o_buf.data_ptr())
                        torch.cuda.synchronize()
                        outs.append(o_buf.numpy().copy())
                qs.advance()
            results[mode] = np.stack(outs)
    for mode in ("pinned", "pageable", "pinned_unaligned"):
        assert np.array_equal(results["device"], results[mode]), mode


def test_segment_pool_exhaustion_reports_capacity():
    w = W.Workload("cap", B=1, L=1, Hq=2, Hkv=2, ctx_len=[64 * 300], topk=8, buf_mult=2,
                   drift_a=0.5, drift_c=0.5, steps=3, seed=29)
    from sparse_attention_tiered_gb300 import SpinContext, SpinError
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_CAPACITY
    with SpinContext.for_workload(w, seg_pool_segments=2) as ctx:
        k, v = w.request_kv(0, 0)
        ctx.index_offload_host(0, 0, k, v)
        q = torch.from_numpy(w.queries().bf16()[0].view(np.int16)).cuda()
        out = torch.empty((1, 2, 128), dtype=torch.float32, device="cuda")
        ctx.decode_step(0, q, out)
        st = ctx.stats(check=False)
        assert st["rc"] == SPIN_ERR_CAPACITY
        with pytest.raises(SpinError):
            ctx.decode_step(0, q, out)


def test_invalid_arguments_and_order():
    from sparse_attention_tiered_gb300 import SpinContext, SpinError
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_INVALID, SPIN_ERR_STATE
    w = W.Workload("inv", B=2, L=1, Hq=4, Hkv=2, ctx_len=[128, 256], topk=2, buf_mult=1,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=0)
    with SpinContext.for_workload(w) as ctx:
        q = torch.zeros((2, 4, 128), dtype=torch.int16, device="cuda")
        out = torch.empty((2, 4, 128), dtype=torch.float32, device="cuda")
        with pytest.raises(SpinError) as e:
            ctx.decode_step(0, q, out)          # nothing offloaded yet
        assert e.value.code == SPIN_ERR_STATE
        with pytest.raises(SpinError) as e:
            ctx.decode_step(1, q, out)          # no such layer
        assert e.value.code == SPIN_ERR_INVALID
        k, v = w.request_kv(0, 0)
        from sparse_attention_tiered_gb300 import spin_index_offload
        with pytest.raises(SpinError) as e:      # wrong token count for request 1
            spin_index_offload(ctx.h, 1, 0, k.ctypes.data, v.ctypes.data, 128, True)
        assert e.value.code == SPIN_ERR_INVALID
        with pytest.raises(SpinError) as e:      # misaligned source
            spin_index_offload(ctx.h, 0, 0, k.ctypes.data + 2, v.ctypes.data, 128, True)
        assert e.value.code == SPIN_ERR_INVALID


# ---------------------------------------------------------------------------
# KV append (tail mode): one token per request and layer before every decode step.
# ---------------------------------------------------------------------------
def test_append_tail_lockstep_narrow():
    """Ragged initial contexts (tails of 40, 17, 2 and 0 tokens, one empty request), GQA 5, two
    layers, 2x buffer: tails fill and become selectable partitions mid-run; the tail page, the
    grown summaries, page state and outputs follow the oracle's tail mode."""
    w = W.Workload("append", B=4, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 130, 0], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=80, seed=21)
    ls = Lockstep(w, append=w.steps)
    try:
        for _ in range(w.steps):
            ls.step()
        st = ls.ctx.stats()
        assert st["device_error"] == 0
        assert st["appended_tokens"] == w.steps * w.B * w.L
        # every request's tail filled at least once (40 + 24, 17 + 47, 2 + 62, 0 + 64 tokens)
        assert st["tail_flushes"] >= w.B * w.L
        assert ls.ctx.P_lb[0] == [(n + w.steps) // 64 for n in w.ctx_len]
        assert ls.report.max_out_err <= OUT_TOL and st["evictions"] > 0
    finally:
        ls.close()


@pytest.mark.parametrize("G", [8, 16])
def test_append_tail_lockstep_wide(G):
    """64 units per layer (the fused score path), GQA 8 and 16 (one and two head tiles)."""
    w = W.Workload("append_wide", B=32, L=1, Hq=2 * G, Hkv=2, ctx_len=[1984 + 13 * b for b in range(32)], topk=6,
                   buf_mult=3, drift_a=0.8, drift_c=0.2, steps=70, seed=43)
    ls = Lockstep(w, append=w.steps, units=sample_units(w, 16, seed=3))
    try:
        for _ in range(w.steps):
            ls.step()
        st = ls.ctx.stats()
        assert st["device_error"] == 0 and st["tail_flushes"] >= w.B
        assert ls.report.max_out_err <= OUT_TOL
    finally:
        ls.close()


def test_append_errors():
    """Append on a fixed-context handle is out of order; growing past ctx_len + append_tokens is
    refused before anything is enqueued, and the context stays usable."""
    from sparse_attention_tiered_gb300 import SpinContext, SpinError
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_CAPACITY, SPIN_ERR_STATE
    w = W.Workload("append_err", B=2, L=1, Hq=4, Hkv=2, ctx_len=[100, 64], topk=2, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=0)
    kn = torch.zeros((2, 2, 128), dtype=torch.int16, device="cuda")
    with SpinContext.for_workload(w) as ctx:
        with pytest.raises(SpinError) as e:
            ctx.append_kv(0, kn, kn)
        assert e.value.code == SPIN_ERR_STATE
    with SpinContext.for_workload(w, append_tokens=2) as ctx:
        for b in range(w.B):
            ctx.index_offload_host(b, 0, *w.request_kv(0, b))
        ctx.append_kv(0, kn, kn)
        ctx.append_kv(0, kn, kn)
        with pytest.raises(SpinError) as e:
            ctx.append_kv(0, kn, kn)
        assert e.value.code == SPIN_ERR_CAPACITY
        q = torch.from_numpy(w.queries().bf16()[0].view(np.int16)).cuda()
        out = torch.empty((2, 4, 128), dtype=torch.float32, device="cuda")
        ctx.decode_step(0, q, out)
        st = ctx.stats()
        assert st["appended_tokens"] == 4 and st["device_error"] == 0
        assert ctx.P_lb[0] == [1, 1] and ctx.tail_lb[0] == [38, 2]


# ---------------------------------------------------------------------------
# Variable partitions: groups of 1..64 tokens, each in a page of its own.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mean_part", [20, 48])
def test_variable_partitions_lockstep_narrow(mean_part):
    """The generator's grouping (tokens shuffled within 256-token windows, groups of 1..64):
    ragged contexts, a request with fewer groups than top-k (every group selected, so the
    output is dense attention over all its tokens), an empty request, GQA 5, 2x buffer.
    Summaries, the first step's resident pages, selections, page state and outputs follow
    the oracle over the same grouping."""
    w = W.Workload("parts", B=4, L=2, Hq=10, Hkv=2, ctx_len=[3000, 777, 100, 0], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=12, seed=51, mean_part=mean_part)
    ls = Lockstep(w)
    try:
        assert ls.ctx.P_lb[1] == [w.var_partitions(b) for b in range(w.B)]
        for _ in range(w.steps):
            ls.step()
        st = ls.ctx.stats()
        assert st["device_error"] == 0 and st["evictions"] > 0
        assert ls.report.max_out_err <= OUT_TOL and ls.report.exact_units > 0
    finally:
        ls.close()


def test_variable_partitions_lockstep_wide():
    """64 units per layer (the fused score path), GQA 8, K/V offloaded from device memory."""
    w = W.Workload("parts_wide", B=32, L=1, Hq=16, Hkv=2, ctx_len=[1500 + 37 * b for b in range(32)], topk=6,
                   buf_mult=3, drift_a=0.8, drift_c=0.2, steps=10, seed=53, mean_part=30)
    rep, st = _run(w, units=sample_units(w, 16, seed=5), offload_from_device=True)
    assert st["evictions"] > 0 and rep.max_out_err <= OUT_TOL


def test_variable_partitions_errors():
    """Each offload entry point refuses the other mode; groupings that break the rules are
    refused before anything is enqueued, and the context stays usable."""
    from sparse_attention_tiered_gb300 import SpinContext, SpinError
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_INVALID, SPIN_ERR_STATE
    w = W.Workload("parts_err", B=1, L=1, Hq=4, Hkv=2, ctx_len=[300], topk=3, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=0, mean_part=30)
    k, v = w.request_kv(0, 0)
    order, starts = w.request_parts(0, 0)
    with SpinContext(w.B, w.L, w.Hq, w.Hkv, w.ctx_len, w.topk, w.buf_mult) as ctx:  # fixed partitions
        with pytest.raises(SpinError) as e:
            ctx.index_offload_parts(0, 0, k, v, order, starts)
        assert e.value.code == SPIN_ERR_STATE
    with SpinContext.for_workload(w) as ctx:
        assert ctx.max_partitions == w.max_partitions == 10
        with pytest.raises(SpinError) as e:
            ctx.index_offload_host(0, 0, k, v)
        assert e.value.code == SPIN_ERR_STATE
        bad = []
        s1 = starts.copy(); s1[0, 1] = 0                          # an empty partition
        bad.append((order, s1))
        s2 = np.array([[0, 65, 300], [0, 150, 300]], np.int32)    # a partition of 65 tokens
        bad.append((order, s2))
        s3 = starts.copy(); s3[1, -1] = 299                       # does not end at n_tokens
        bad.append((order, s3))
        o4 = order.copy(); o4[0, 5] = o4[0, 6]                     # a token twice
        bad.append((o4, starts))
        o5 = order.copy(); o5[1, 0] = 300                          # a token out of range
        bad.append((o5, starts))
        s6 = np.tile(np.arange(0, 301, 25, dtype=np.int32), (2, 1))  # 12 partitions > max_partitions
        bad.append((order, s6))
        for o_, s_ in bad:
            with pytest.raises(SpinError) as e:
                ctx.index_offload_parts(0, 0, k, v, o_, s_)
            assert e.value.code == SPIN_ERR_INVALID
        q = torch.from_numpy(w.queries().bf16()[0].view(np.int16)).cuda()
        out = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
        with pytest.raises(SpinError) as e:  # nothing was offloaded
            ctx.decode_step(0, q, out)
        assert e.value.code == SPIN_ERR_STATE
        ctx.index_offload_parts(0, 0, k, v, order, starts)
        ctx.decode_step(0, q, out)
        assert ctx.stats()["device_error"] == 0 and torch.isfinite(out).all()


# ---------------------------------------------------------------------------
# Buffer elasticity: per-request budgets change between steps.
# ---------------------------------------------------------------------------
def test_buffer_elasticity_lockstep():
    """Budgets shrink to the mandatory pages, grow back and shrink again on different
    requests mid-run; page state stays bit-exact with the oracle and no unit keeps more
    pages resident than its request's budget."""
    w = W.Workload("elastic", B=3, L=2, Hq=10, Hkv=2, ctx_len=[3000, 4113, 9000], topk=8, buf_mult=4,
                   drift_a=0.8, drift_c=0.2, steps=30, seed=53)
    events = {8: [(0, 8), (2, 16)], 16: [(0, 32)], 22: [(1, 8), (2, 9)]}
    ls = Lockstep(w, budgets=events)
    try:
        for _ in range(w.steps):
            ls.step()
        st = ls.ctx.stats()
        assert st["device_error"] == 0 and st["evictions"] > 0
        assert ls.report.max_out_err <= OUT_TOL
        from sparse_attention_tiered_gb300 import SpinError
        from sparse_attention_tiered_gb300._binding import SPIN_ERR_INVALID
        for b, pages in ((0, w.topk - 1), (0, w.cap + 1), (w.B, w.topk)):
            with pytest.raises(SpinError) as e:
                ls.ctx.set_buffer(b, pages)
            assert e.value.code == SPIN_ERR_INVALID
    finally:
        ls.close()


# ---------------------------------------------------------------------------
# Full-size workloads: every unit against the oracle, every step, in the launch
# configuration the benchmark times.
# ---------------------------------------------------------------------------
FULL = ["qwen3_14b_32k", "llama31_70b_128k", "stress_m1", "stress_m5", "long_1m"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_all_units(name):
    w = W.by_name(name)
    h = AllUnits(w)
    try:
        for _ in range(w.steps):
            h.step()
        st = h.ctx.stats()
        assert st["device_error"] == 0
    finally:
        h.close()
    rep = h.report
    print(f"\n{name}: {rep.exact_units}/{rep.compared_units} unit-steps exact, {rep.tie_divergences} tie-band "
          f"divergences, max out err {rep.max_out_err:.3e}, evictions {rep.evictions}, misses {rep.misses}")
    assert rep.compared_units == w.units * w.steps
    assert rep.exact_units >= 0.99 * rep.compared_units, rep.notes[:10]
    assert rep.max_out_err <= OUT_TOL
    if name.startswith("stress"):
        assert st["evictions"] > 0 and rep.evictions > 0


def test_bounded_wait_reports_timeout():
    """Failure detection without a GPU fault: with the retriever warps disabled nothing ever
    publishes a missing page, so the producer's bounded wait runs out (about 2 s); the step
    finishes, the device error word says so, and the context keeps reporting SPIN_ERR_TIMEOUT."""
    import time
    from sparse_attention_tiered_gb300 import SpinContext, SpinError
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_TIMEOUT, SPIN_FLAG_TEST_NO_RETRIEVE
    w = W.Workload("timeout", B=1, L=1, Hq=4, Hkv=2, ctx_len=[64 * 40], topk=4, buf_mult=2,
                   drift_a=0.9, drift_c=0.1, steps=1, seed=37)
    with SpinContext.for_workload(w, flags=SPIN_FLAG_TEST_NO_RETRIEVE) as ctx:
        k, v = w.request_kv(0, 0)
        ctx.index_offload_host(0, 0, k, v)
        q = torch.from_numpy(w.queries().bf16()[0].view(np.int16)).cuda()
        out = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
        t0 = time.time()
        ctx.decode_step(0, q, out)
        st = ctx.stats(check=False)
        assert st["rc"] == SPIN_ERR_TIMEOUT and st["device_error"] & 2
        assert time.time() - t0 < 60
        with pytest.raises(SpinError) as e:
            ctx.decode_step(0, q, out)
        assert e.value.code == SPIN_ERR_TIMEOUT
    # the CUDA context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def test_tier_split_metadata_same_results_less_hbm():
    """Second-level segments in pinned host memory: identical lockstep results, and the
    page metadata left in HBM shrinks by the segment pool."""
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_TIER_SPLIT
    w = W.Workload("tier", B=3, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 9000], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=16, seed=41)
    rep_a, st_a = _run(w)
    rep_b, st_b = _run(w, flags=SPIN_FLAG_TIER_SPLIT)
    assert rep_b.max_out_err <= OUT_TOL and rep_b.evictions == rep_a.evictions
    for key in ("hits", "misses", "evictions", "live_segments"):
        assert st_a[key] == st_b[key], key
    assert st_b["metadata_bytes"] == st_a["metadata_bytes"] - st_a["pool_segments"] * 64 * 4


def test_metadata_accounting_flat_worst_case():
    """The flat table of the pages' worst-case logical space (one int32 per partition of
    max_context, per request, layer and KV head, plus the per-page state) against the
    two-level table's directory (covering max_context), segment pool, live counts, bitmap
    and the same per-page state; identical results with and without the larger directory."""
    w = W.Workload("meta", B=3, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 9000], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=6, seed=41)
    rep_a, st_a = _run(w)
    wl = w.with_(max_context=65536)
    rep_b, st_b = _run(wl)
    for key in ("hits", "misses", "evictions", "live_segments"):
        assert st_a[key] == st_b[key], key
    units, slots = w.units, w.units * w.cap
    S = st_b["pool_segments"]
    Dl = -(-(65536 // 64) // 64)
    assert st_b["flat_table_bytes"] == (units * (65536 // 64) + 2 * slots) * 4
    assert st_b["metadata_bytes"] == (units * Dl + S * 64 + S + (S + 31) // 32 + 2 * slots) * 4
    assert st_b["flat_table_bytes"] > st_b["metadata_bytes"]
    P_max = max(w.partitions(b) for b in range(w.B))
    assert st_a["flat_table_bytes"] == (units * P_max + 2 * slots) * 4


def test_phased_kernel_same_results():
    """The phased decode-step kernel (scoring, then managing, then retrieval over the whole
    grid) against the pipelined one this workload gets by default: both in lockstep with
    the oracle, with the same paging record."""
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_PHASED
    w = W.Workload("phased", B=5, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 9000, 64, 0], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=12, seed=59)
    rep_a, st_a = _run(w)
    rep_b, st_b = _run(w, flags=SPIN_FLAG_PHASED)
    assert rep_a.max_out_err <= OUT_TOL and rep_b.max_out_err <= OUT_TOL
    for key in ("hits", "misses", "evictions", "lru_rounds", "live_segments"):
        assert st_a[key] == st_b[key], key


def test_hugepage_host_store_same_results():
    """The page store as a huge-page mapping registered with CUDA: identical lockstep results."""
    from sparse_attention_tiered_gb300._binding import SPIN_FLAG_HOST_HUGEPAGES
    w = W.Workload("huge", B=3, L=2, Hq=10, Hkv=2, ctx_len=[1000, 4113, 9000], topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=12, seed=47)
    rep_a, st_a = _run(w)
    rep_b, st_b = _run(w, flags=SPIN_FLAG_HOST_HUGEPAGES)
    assert rep_b.max_out_err <= OUT_TOL
    for key in ("hits", "misses", "evictions", "live_segments", "host_store_bytes"):
        assert st_a[key] == st_b[key], key


def _wide_ties_run(P, npat, scale_spread, topk, steps, seed):
    """One unit with P partitions copied from `npat` patterns (exact score ties between
    copies), scaled over `scale_spread` binades; GPU vs oracle every step."""
    from sparse_attention_tiered_gb300 import SpinContext
    rng = np.random.default_rng(seed)
    G, cap = 2, 2 * topk
    pat_k = rng.standard_normal((npat, 64, 128)).astype(np.float32)
    pat_v = rng.standard_normal((npat, 64, 128)).astype(np.float32)
    scales = 2.0 ** (np.arange(npat) % max(scale_spread, 1))
    pat_k *= scales[:, None, None]
    to_bits = lambda x: (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kp, vp = to_bits(pat_k), to_bits(pat_v)
    idx = np.arange(P) % npat
    k = np.ascontiguousarray(kp[idx].reshape(1, P * 64, 128))
    v = np.ascontiguousarray(vp[idx].reshape(1, P * 64, 128))
    ctx = SpinContext(1, 1, G, 1, [P * 64], topk, 2)
    try:
        ctx.index_offload_host(0, 0, k, v)
        torch.cuda.synchronize()
        u = O.Unit(P * 64, cap, k[0], v[0])
        out = torch.empty((1, G, 128), dtype=torch.float32, device="cuda")
        for t in range(steps):
            qf = rng.standard_normal((G, 128)).astype(np.float32)
            qb = to_bits(qf)
            ctx.decode_step(0, torch.from_numpy(qb.view(np.int16)[None]).cuda(), out)
            torch.cuda.synchronize()
            r = u.step(qb, topk, t)
            ex = ctx.export(0)
            keff = int(ex["keff"][0])
            assert np.array_equal(ex["sel"][0][:keff], r["sel"]), f"step {t}: selection differs"
            assert np.array_equal(ex["sel_slot"][0][:keff], r["sel_slot"]), f"step {t}: slots differ"
            err = float(np.abs(out.cpu().numpy()[0] - r["out"]).max())
            assert err <= OUT_TOL, f"step {t}: output error {err}"
        assert ctx.stats()["device_error"] == 0
    finally:
        ctx.close()


def test_wide_unit_exact_ties_candidate_and_list_paths():
    """P > 4096: 100 exact copies of each of 50 patterns spread over 12 binades; the k-th
    largest score sits in a tie group, resolved to the lowest partitions."""
    _wide_ties_run(P=5000, npat=50, scale_spread=12, topk=64, steps=4, seed=61)


@pytest.mark.parametrize("P,npat,topk", [(512, 20, 32), (300, 3, 20), (512, 1, 32), (130, 7, 32)])
def test_small_unit_exact_ties(P, npat, topk):
    """Small units (P <= 512, k <= 32, the manager groups of 128 threads): exact score
    ties within and across warps' slices of the keys, resolved to the lowest partitions,
    GPU against the oracle every step."""
    _wide_ties_run(P=P, npat=npat, scale_spread=4, topk=topk, steps=3, seed=71 + P)


def test_wide_unit_all_equal_scores_fallbacks():
    """P > 4096, every partition identical: more tied keys than either list holds, so the
    full-scan radix passes and the warp-scan compaction run; partitions 0..k-1 win."""
    _wide_ties_run(P=5000, npat=1, scale_spread=1, topk=64, steps=2, seed=67)
