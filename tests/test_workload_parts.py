"""The seeded grouping behind variable partitions (an input generator, no method arithmetic):
every head's order is a permutation, groups hold 1..64 tokens, counts follow the rule, the
draw is reproducible and independent per unit."""
import numpy as np
import pytest

import workload as W


@pytest.mark.parametrize("n,P", [(1, 1), (64, 1), (65, 2), (300, 7), (4096, 64), (4096, 4096), (5000, 171)])
def test_random_parts_shape_rules(n, P):
    rng = np.random.default_rng(n * 31 + P)
    order, starts = W.random_parts(rng, n, P)
    assert order.dtype == np.int32 and starts.dtype == np.int32
    assert sorted(order.tolist()) == list(range(n))
    sizes = np.diff(starts)
    assert starts[0] == 0 and starts[-1] == n and len(sizes) == P
    assert sizes.min() >= 1 and sizes.max() <= 64
    # tokens move only within their 256-token window
    assert np.all(order // 256 == np.arange(n) // 256)


def test_random_parts_empty_and_impossible():
    order, starts = W.random_parts(np.random.default_rng(0), 0, 0)
    assert order.size == 0 and starts.tolist() == [0]
    with pytest.raises(AssertionError):
        W.random_parts(np.random.default_rng(0), 129, 2)  # 2 groups cannot hold 129 tokens


def test_workload_grouping_counts_and_reproducibility():
    w = W.Workload("g", B=3, L=2, Hq=4, Hkv=2, ctx_len=[1000, 64, 0], topk=4, buf_mult=2, drift_a=0.9,
                   drift_c=0.1, steps=1, seed=7, mean_part=20)
    assert [w.var_partitions(b) for b in range(3)] == [50, 4, 0]
    assert w.max_partitions == 50
    # at least ceil(ctx / 64) groups even when the mean asks for fewer
    assert w.with_(mean_part=1000).var_partitions(0) == 16
    o1, s1 = w.request_parts(1, 0)
    o2, s2 = w.request_parts(1, 0)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    assert o1.shape == (2, 1000) and s1.shape == (2, 51)
    # units draw independently: heads and layers differ
    assert not np.array_equal(o1[0], o1[1])
    assert not np.array_equal(w.request_parts(0, 0)[0], o1)
    # the seed changes the draw
    assert not np.array_equal(w.with_(seed=8).request_parts(1, 0)[0], o1)
