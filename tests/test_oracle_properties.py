"""Property tests of the oracle over randomized inputs (hypothesis): the same pins as
oracle_pins.py, driven over many more sizes, ties, groupings and budget schedules."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle as O  # noqa: E402
import oracle_pins as pins  # noqa: E402
import workload as W  # noqa: E402

SETTINGS = dict(max_examples=120, deadline=None, derandomize=True)


@settings(**SETTINGS)
@given(P=st.integers(1, 11), k=st.integers(1, 13), levels=st.integers(1, 5), seed=st.integers(0, 2**31 - 1))
def test_topk_matches_brute_force_with_ties(P, k, levels, seed):
    rng = np.random.default_rng(seed)
    sc = rng.integers(0, levels, size=P).astype(np.float64)  # few distinct values: many exact ties
    assert list(O.topk(sc, k)) == pins.brute_topk(sc, k)


@settings(**SETTINGS)
@given(ntok=st.integers(1, 64 * 40), frac=st.floats(0.05, 1.0), mult=st.integers(1, 4), steps=st.integers(1, 12),
       locality=st.floats(0.0, 1.0), seed=st.integers(0, 2**31 - 1))
def test_manager_invariants_random_runs(ntok, frac, mult, steps, locality, seed):
    P = (ntok + 63) // 64
    k = max(1, int(round(frac * P)))
    pins._run_invariants(O.load(), ntok, cap=mult * k, k=k, steps=steps, seed=seed, locality=locality)


@settings(**SETTINGS)
@given(ntok=st.integers(64, 64 * 24), mult=st.integers(2, 4), seed=st.integers(0, 2**31 - 1),
       changes=st.lists(st.tuples(st.integers(1, 10), st.floats(0.0, 1.0)), max_size=4))
def test_manager_invariants_with_budget_changes(ntok, mult, seed, changes):
    P = (ntok + 63) // 64
    k = max(1, P // 4)
    cap = mult * k
    budgets = {t: k + int(round(f * (cap - k))) for t, f in changes}
    pins._run_invariants(O.load(), ntok, cap=cap, k=k, steps=12, seed=seed, locality=0.6, budgets=budgets)


@settings(**SETTINGS)
@given(n=st.integers(1, 700), per=st.floats(1.0, 64.0), seed=st.integers(0, 2**31 - 1))
def test_variable_partition_index_and_dense_identity(n, per, seed):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(seed)
    P = min(n, max(-(-n // 64), int(round(n / per))))
    order, starts = W.random_parts(rng, n, P)
    k, v = pins.rand_kv(rng, n, scale=1.3)
    summ = O.index_parts(k, order, starts)
    kf = pins.bf(k)
    ref = np.stack([kf[order[starts[p]:starts[p + 1]]].mean(axis=0) for p in range(P)])
    assert np.abs(summ - ref).max() <= 1e-12
    G = 1 + seed % 4
    q = pins.f32_to_bf16_bits(rng.standard_normal((G, 128)).astype(np.float32))
    u = O.Unit.from_parts(k, v, order, starts, cap=P)
    out = u.step(q, k=P, t=0)["out"]
    qt = torch.from_numpy(pins.bf(q)).view(1, G, 1, 128)
    kt = torch.from_numpy(kf).view(1, 1, n, 128).expand(1, G, n, 128)
    vt = torch.from_numpy(pins.bf(v)).view(1, 1, n, 128).expand(1, G, n, 128)
    dense = F.scaled_dot_product_attention(qt, kt, vt).view(G, 128).numpy()
    assert np.abs(out - dense).max() <= 1e-12
