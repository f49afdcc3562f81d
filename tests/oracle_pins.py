"""Pins of the oracle to facts outside itself.

Each ``check_*`` takes an oracle library handle and raises AssertionError when
the oracle disagrees with a closed form, a library routine, a brute-force
enumeration or an invariant of the method. ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutations.py`` runs them on oracle builds with a
planted mistake and expects at least one of them to fail.

What pins what:
  attention   dense identity (top-k = all partitions equals plain softmax
              attention computed by torch's scaled_dot_product_attention in
              float64); 1-token and equal-key closed forms
  scores      coordinate probe (q = e_i on every head gives G * summary[i])
  top-k       brute force over all k-subsets with the equal-score rule
  index       constant partitions, ragged tail, and recovery of the drawn
              per-partition offsets within the sampling error 1/8
  manage      bucketed-LRU invariants, page-table round trip, slot-order rule,
              a hand-traced scenario
  retrieve    byte equality of resident pages with the host pages
  variable    partitions given as a token order and boundaries: numpy means of
  partitions  the gathered rows, single-token and constant groups, page rows in
              order with zero padding, dense identity over all tokens whatever
              the grouping, and a partial selection equal to dense attention
              over the union of the chosen groups' tokens
"""
from __future__ import annotations

import itertools

import numpy as np

import oracle as O
import workload as W

D, PART = 128, 64


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits (used to build exact test inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf(bits: np.ndarray) -> np.ndarray:
    return W.bf16_to_f64(bits)


def rand_kv(rng, ntok, scale=1.0):
    k = f32_to_bf16_bits(rng.standard_normal((ntok, D)).astype(np.float32) * scale)
    v = f32_to_bf16_bits(rng.standard_normal((ntok, D)).astype(np.float32))
    return k, v


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def check_dense_attention(lib):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(1)
    for ntok, G in ((200, 3), (64, 1), (1000, 8), (130, 5)):
        k, v = rand_kv(rng, ntok, scale=1.5)
        P = (ntok + PART - 1) // PART
        u = O.Unit(ntok, cap=P, k_bits=k, v_bits=v, lib=lib)
        q = f32_to_bf16_bits(rng.standard_normal((G, D)).astype(np.float32))
        r = u.step(q, k=P, t=0)
        assert list(r["sel"]) == list(range(P)), "top-k = P must select every partition"
        qt = torch.from_numpy(bf(q)).view(1, G, 1, D)
        kt = torch.from_numpy(bf(k)).view(1, 1, ntok, D).expand(1, G, ntok, D)
        vt = torch.from_numpy(bf(v)).view(1, 1, ntok, D).expand(1, G, ntok, D)
        ref = F.scaled_dot_product_attention(qt, kt, vt).view(G, D).numpy()
        err = np.abs(r["out"] - ref).max()
        assert err <= 1e-12, f"dense identity broken (ntok={ntok}, G={G}): max err {err}"


def check_attention_closed_forms(lib):
    rng = np.random.default_rng(2)
    # one token: the output is that token's value
    k, v = rand_kv(rng, 1)
    u = O.Unit(1, cap=1, k_bits=k, v_bits=v, lib=lib)
    q = f32_to_bf16_bits(rng.standard_normal((2, D)).astype(np.float32))
    r = u.step(q, k=1, t=0)
    assert np.array_equal(r["out"], np.repeat(bf(v), 2, axis=0)), "1-token attention must return v"
    # identical keys: softmax is uniform, the output is the mean value row
    ntok = 150
    krow = f32_to_bf16_bits(rng.standard_normal((1, D)).astype(np.float32))
    k = np.repeat(krow, ntok, axis=0)
    _, v = rand_kv(rng, ntok)
    u = O.Unit(ntok, cap=3, k_bits=k, v_bits=v, lib=lib)
    r = u.step(q, k=3, t=0)
    mean_v = bf(v).mean(axis=0)
    assert np.abs(r["out"] - mean_v[None, :]).max() < 1e-12, "equal keys must average the values"


# ---------------------------------------------------------------------------
# scores and top-k
# ---------------------------------------------------------------------------

def check_scores_probe(lib):
    """q = e_i on every head of a G-group scores partition p as G * summary_p[i]."""
    rng = np.random.default_rng(3)
    P, G = 7, 3
    summ = rng.standard_normal((P, D))
    for i in (0, 5, 127):
        q = np.zeros((G, D), np.uint16)
        q[:, i] = 0x3F80  # bf16 1.0
        sc = O.scores(summ, q, lib)
        assert np.array_equal(sc, G * summ[:, i]), f"score probe failed for coordinate {i}"
    # a single head with a two-hot query picks two coordinates with their weights
    q = np.zeros((1, D), np.uint16)
    q[0, 3] = 0x4000   # 2.0
    q[0, 9] = 0xBF00   # -0.5
    sc = O.scores(summ, q, lib)
    assert np.array_equal(sc, 2.0 * summ[:, 3] - 0.5 * summ[:, 9])


def brute_topk(sc, k):
    """All k-subsets; the chosen one is ranked first by scores (desc) then indices (asc)."""
    P = len(sc)
    k = min(k, P)
    best = None
    for comb in itertools.combinations(range(P), k):
        key = sorted(((-sc[p], p) for p in comb))
        if best is None or key < best[0]:
            best = (key, comb)
    return sorted(best[1])


def check_topk_bruteforce(lib):
    rng = np.random.default_rng(4)
    for trial in range(60):
        P = int(rng.integers(1, 13))
        k = int(rng.integers(1, 14))
        # integer-valued scores force many exact ties
        sc = rng.integers(-3, 4, size=P).astype(np.float64)
        if trial % 3 == 0:
            sc = rng.standard_normal(P)
        got = list(O.topk(sc, k, lib))
        assert got == brute_topk(sc, k), f"top-k mismatch P={P} k={k} sc={sc} got={got}"
    # ties by duplicated summaries through the full scoring path
    summ = np.repeat(rng.standard_normal((3, D)), 4, axis=0)   # partitions 0-3, 4-7, 8-11 identical
    q = f32_to_bf16_bits(rng.standard_normal((2, D)).astype(np.float32))
    sc = O.scores(summ, q, lib)
    for k in (1, 2, 5, 6, 11):
        assert list(O.topk(sc, k, lib)) == brute_topk(sc, k)


# ---------------------------------------------------------------------------
# index
# ---------------------------------------------------------------------------

def check_index(lib):
    rng = np.random.default_rng(5)
    ntok = 64 * 3 + 17                     # ragged tail: 17 tokens in the last partition
    P = 4
    consts = f32_to_bf16_bits(rng.standard_normal((P, D)).astype(np.float32))
    k = np.empty((ntok, D), np.uint16)
    for p in range(P):
        k[p * PART:min((p + 1) * PART, ntok)] = consts[p]
    s = O.index(k, lib)
    assert np.array_equal(s, bf(consts)), "mean of a constant partition must be the constant"
    # mean over exactly the valid tokens of the tail: rows 192..208 hold 0..16
    k2 = np.zeros((ntok, D), np.uint16)
    vals = np.arange(17, dtype=np.float32)
    k2[192:] = f32_to_bf16_bits(np.repeat(vals[:, None], D, axis=1))
    s2 = O.index(k2, lib)
    assert np.allclose(s2[3], 8.0, atol=0, rtol=0), "tail mean must divide by its valid tokens"
    # drawn offsets come back within the sampling error of a 64-token mean (std 1/8)
    w = W.tiny()
    kb, _ = w.unit_kv(0, 0, 2)
    mu = w.unit_mu(0, 0, 2).astype(np.float64)
    err = O.index(kb, lib) - mu
    assert abs(err.std() - 0.125) < 0.0125 and abs(err.mean()) < 0.005, (err.std(), err.mean())


# ---------------------------------------------------------------------------
# manage / retrieve
# ---------------------------------------------------------------------------

def _bucket(t, last):
    return 63 - min(63, t - last)


def _run_invariants(lib, ntok, cap, k, steps, seed, locality, budgets=None):
    rng = np.random.default_rng(seed)
    kb, vb = rand_kv(rng, ntok)
    u = O.Unit(ntok, cap=cap, k_bits=kb, v_bits=vb, lib=lib)
    P = u.P
    budget = cap
    prev = np.sort(rng.choice(P, size=min(k, P), replace=False))
    for t in range(steps):
        if budgets and t in budgets:
            budget = budgets[t]
            u.set_budget(budget)
        # a selection that keeps part of the previous one (temporal locality)
        keep = prev[rng.random(prev.size) < locality]
        fresh = rng.choice(P, size=min(k, P), replace=False)
        pool = list(dict.fromkeys(list(keep) + list(fresh)))
        sel = np.sort(np.array(pool[:min(k, P)], np.int32))
        sp0, lu0, rs0 = u.export()
        resident0 = {int(p) for p in sp0 if p >= 0}
        sel_slot, sel_hit, victims, mo = u.manage(sel, t)
        sp1, lu1, rs1 = u.export()
        # hits are exactly the selected partitions resident before the step
        assert [bool(int(p) in resident0) for p in sel] == list(sel_hit)
        assert mo.hits == int(sel_hit.sum()) and mo.misses == len(sel) - mo.hits
        free0 = budget - len(resident0)
        demand = mo.misses - free0
        assert mo.demand == demand
        mand = set(int(p) for p in sel)
        if demand <= 0:
            assert mo.evicted == 0 and mo.cutoff == -1
        else:
            assert mo.evicted >= demand, "evicted must cover the demand"
            assert not (set(int(v) for v in victims) & mand), "a mandatory page was evicted"
            # buckets are taken from the timestamps before the step
            nm = [(s, int(sp0[s])) for s in range(cap) if sp0[s] >= 0 and int(sp0[s]) not in mand]
            bucket = {p: _bucket(t, int(lu0[s])) for s, p in nm}
            vset = set(int(v) for v in victims)
            for s, p in nm:
                if bucket[p] <= mo.cutoff:
                    assert p in vset, "a page in a reclaimed bucket survived"
                else:
                    assert p not in vset, "a page above the cutoff bucket was evicted"
            below = sum(1 for _, p in nm if bucket[p] < mo.cutoff)
            assert below < demand, "cutoff bucket is not the smallest that covers the demand"
            # victims listed in ascending slot order
            vs = [s for s, p in nm if p in vset]
            assert [int(sp0[s]) for s in vs] == [int(v) for v in victims]
        # every selected partition is resident afterwards, with timestamp t
        assert len(set(sel_slot.tolist())) == len(sel)
        for p, s in zip(sel, sel_slot):
            assert sp1[s] == p and lu1[s] == t and rs1[p] == s
        # misses took the lowest free slots, ascending partition -> ascending slot
        free_after_evict = sorted(s for s in range(cap) if sp0[s] < 0 or int(sp0[s]) in set(map(int, victims)))
        miss_slots = [int(s) for s, h in zip(sel_slot, sel_hit) if not h]
        assert miss_slots == free_after_evict[:len(miss_slots)]
        # resident <= budget <= cap; page table round trip; live segments = occupied 64-ranges
        res = [int(p) for p in sp1 if p >= 0]
        assert len(res) <= budget <= cap and len(set(res)) == len(res)
        for p in range(P):
            s = rs1[p]
            if s >= 0:
                assert sp1[s] == p
            else:
                assert p not in res
        assert u.live_segments() == len({p // 64 for p in res})
        # retrieve: resident pages equal the host pages byte for byte
        for p, s in zip(sel, sel_slot):
            page = u.slot_page(int(s))
            exp_k = np.zeros((PART, D), np.uint16)
            exp_v = np.zeros((PART, D), np.uint16)
            rows = kb[p * PART:(p + 1) * PART]
            exp_k[:rows.shape[0]] = rows
            exp_v[:rows.shape[0]] = vb[p * PART:(p + 1) * PART]
            assert np.array_equal(page[0], exp_k) and np.array_equal(page[1], exp_v)
        prev = sel
    return u


def check_lru_invariants(lib):
    _run_invariants(lib, ntok=300 * 64 + 5, cap=8, k=4, steps=150, seed=6, locality=0.6)
    _run_invariants(lib, ntok=300 * 64, cap=4, k=4, steps=80, seed=7, locality=0.5)     # no buffering
    _run_invariants(lib, ntok=40 * 64, cap=40, k=8, steps=90, seed=8, locality=0.8)      # cap = P
    _run_invariants(lib, ntok=5 * 64, cap=10, k=8, steps=20, seed=9, locality=0.3)       # k > P
    # buffer elasticity: the budget shrinks to the mandatory pages, grows, shrinks again
    _run_invariants(lib, ntok=300 * 64, cap=20, k=4, steps=120, seed=11, locality=0.7,
                    budgets={30: 4, 50: 20, 80: 9, 100: 5})


def check_budget_hand_trace(lib):
    """Buffer elasticity, hand traced: cap 6, k 2.

    t=0..2 select {0,1}, {2,3}, {4,5}: six misses fill slots 0..5 (last use 0,0,1,1,2,2).
    budget -> 3.
    t=3 sel {5,10}: hit 5 (slot 5, stamped 3), miss 10. resident 6 > budget 3: free -3,
                    demand 1 + 3 = 4. Non-mandatory buckets: 0,1 age 3 -> 60; 2,3 age 2
                    -> 61; 4 age 1 -> 62. Cumulative 2, 4: cutoff 61 reclaims 0,1,2,3
                    (slots 0..3); 10 takes slot 0. Resident {10,4,5} = 3 pages.
    budget -> 6.
    t=4 sel {6,7}: two misses, resident 3, free 3, demand -1: no eviction; slots 1, 2.
    """
    ntok = 20 * 64
    rng = np.random.default_rng(13)
    kb, vb = rand_kv(rng, ntok)
    u = O.Unit(ntok, cap=6, k_bits=kb, v_bits=vb, lib=lib)
    for t, sel in enumerate(([0, 1], [2, 3], [4, 5])):
        ss, hit, vic, mo = u.manage(np.array(sel, np.int32), t)
        assert mo.evicted == 0
    u.set_budget(3)
    ss, hit, vic, mo = u.manage(np.array([5, 10], np.int32), 3)
    assert list(hit) == [True, False] and mo.free_before == -3 and mo.demand == 4 and mo.cutoff == 61
    assert sorted(vic.tolist()) == [0, 1, 2, 3] and list(ss) == [5, 0]
    sp, lu, rs = u.export()
    assert list(sp) == [10, -1, -1, -1, 4, 5] and lu[0] == 3 and lu[5] == 3
    u.set_budget(6)
    ss, hit, vic, mo = u.manage(np.array([6, 7], np.int32), 4)
    assert mo.demand == -1 and mo.evicted == 0 and list(ss) == [1, 2]


def check_lru_hand_trace(lib):
    """Hand-traced scenario: cap 4, k 2, partitions spread over two 64-ranges.

    t=0 sel {1,70}:   misses 2, free 4 -> slots 0,1 (1->0, 70->1); segments: ranges 0 and 1.
    t=1 sel {2,3}:    misses 2, free 2 -> slots 2,3; pages 1,70 keep last_use 0.
    t=2 sel {2,80}:   hit 2 (slot 2); miss 80; free 0, demand 1. Buckets of non-mandatory
                      pages: 1,70 age 2 -> bucket 61; 3 age 1 -> bucket 62. Cutoff 61
                      reclaims both 1 and 70 (slots 0,1); 80 takes slot 0.
                      Range 1 loses 70 then gains 80: still one live segment there.
    t=3 sel {3,5}:    hit 3 (slot 3), miss 5; resident {80,2,3} -> free 1, demand 0;
                      5 takes slot 1.
    """
    ntok = 100 * 64
    rng = np.random.default_rng(10)
    kb, vb = rand_kv(rng, ntok)
    u = O.Unit(ntok, cap=4, k_bits=kb, v_bits=vb, lib=lib)
    ss, hit, vic, mo = u.manage(np.array([1, 70], np.int32), 0)
    assert list(ss) == [0, 1] and not hit.any() and mo.evicted == 0 and u.live_segments() == 2
    ss, hit, vic, mo = u.manage(np.array([2, 3], np.int32), 1)
    assert list(ss) == [2, 3] and mo.demand == 0
    ss, hit, vic, mo = u.manage(np.array([2, 80], np.int32), 2)
    assert list(hit) == [True, False] and mo.demand == 1 and mo.cutoff == 61
    assert sorted(vic.tolist()) == [1, 70] and list(ss) == [2, 0]
    assert u.live_segments() == 2 and u.resolve(1) == -1 and u.resolve(70) == -1 and u.resolve(80) == 0
    ss, hit, vic, mo = u.manage(np.array([3, 5], np.int32), 3)
    assert list(hit) == [True, False] and mo.demand == 0 and list(ss) == [3, 1]
    sp, lu, rs = u.export()
    assert list(sp) == [80, 5, 2, 3] and list(lu) == [2, 3, 2, 3]


def check_step_consistency(lib):
    """The one-call step equals Select -> Manage -> Attend called piecewise."""
    w = W.tiny()
    kb, vb = w.unit_kv(0, 0, 1)
    a = O.Unit(kb.shape[0], cap=w.cap, k_bits=kb, v_bits=vb, lib=lib)
    b = O.Unit(kb.shape[0], cap=w.cap, k_bits=kb, v_bits=vb, lib=lib)
    qs = w.queries()
    for t in range(6):
        q = qs.bf16()[0, 0, 1:2]
        r = a.step(q, w.topk, t)
        sel = O.topk(O.scores(b.summ, q, lib), w.topk, lib)
        ss, hit, vic, mo = b.manage(sel, t)
        out = b.attend(sel, ss, q)
        assert np.array_equal(r["sel"], sel) and np.array_equal(r["sel_slot"], ss)
        assert np.array_equal(r["out"], out)
        qs.advance()
    # the threaded many-unit driver (CPU timing) gives each unit its own one-call step
    units = [O.Unit(kb.shape[0], cap=w.cap, k_bits=kb, v_bits=vb, lib=lib) for _ in range(3)]
    ref = O.Unit(kb.shape[0], cap=w.cap, k_bits=kb, v_bits=vb, lib=lib)
    qs = w.queries()
    for t in range(3):
        q = qs.bf16()[0, 0, 1:2]
        _, keep = O.step_units_parallel(units, [q] * 3, w.topk, t, threads=2, lib=lib)
        r = ref.step(q, w.topk, t)
        for (_, sel, _, _, out) in keep:
            assert np.array_equal(sel[:len(r["sel"])], r["sel"]) and np.array_equal(out, r["out"])
        qs.advance()


def check_append_tail(lib):
    """KV append (tail mode): the tail is attended; with every complete partition selected
    the output is dense attention over all tokens (torch SDPA, float64); appending tokens
    one by one gives the same state as building the unit from all of them; a tail-only
    unit attends its tail."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(12)
    for n0, n_app, G in ((200, 90, 3), (30, 20, 2), (128, 64, 5)):
        n = n0 + n_app
        k, v = rand_kv(rng, n, scale=1.3)
        q = f32_to_bf16_bits(rng.standard_normal((G, D)).astype(np.float32))
        a = O.TailUnit(k[:n0], v[:n0], cap=8, append_max=n_app, lib=lib)
        for r in range(n0, n):
            a.append(k[r], v[r])
        b = O.TailUnit(k, v, cap=8, append_max=0, lib=lib)
        assert a.P == b.P == n // 64 and a.tail_n == b.tail_n == n % 64
        assert np.array_equal(a.summ, b.summ) and np.array_equal(a.host_pages, b.host_pages)
        assert np.array_equal(a.tail[:, :a.tail_n], b.tail[:, :b.tail_n])
        ra = a.step(q, k=max(a.P, 1), t=0)
        rb = b.step(q, k=max(b.P, 1), t=0)
        assert np.array_equal(ra["out"], rb["out"])
        qt = torch.from_numpy(bf(q)).view(1, G, 1, D)
        kt = torch.from_numpy(bf(k)).view(1, 1, n, D).expand(1, G, n, D)
        vt = torch.from_numpy(bf(v)).view(1, 1, n, D).expand(1, G, n, D)
        ref = F.scaled_dot_product_attention(qt, kt, vt).view(G, D).numpy()
        assert np.abs(ra["out"] - ref).max() <= 1e-12, "tail mode must attend every token once"
        # partitions created by appends resolve through the table like the others: the same
        # query again hits every page it just retrieved
        ra2 = a.step(q, k=max(a.P, 1), t=1)
        assert ra2["mo"].hits == min(max(a.P, 1), a.P) == len(ra2["sel"]) and ra2["mo"].misses == 0


def _sdpa(q_bits, k_rows, v_rows):
    import torch
    import torch.nn.functional as F
    G, n = q_bits.shape[0], k_rows.shape[0]
    qt = torch.from_numpy(bf(q_bits)).view(1, G, 1, D)
    kt = torch.from_numpy(bf(k_rows)).view(1, 1, n, D).expand(1, G, n, D)
    vt = torch.from_numpy(bf(v_rows)).view(1, 1, n, D).expand(1, G, n, D)
    return F.scaled_dot_product_attention(qt, kt, vt).view(G, D).numpy()


def check_variable_partitions(lib):
    """Variable partitions: Index, Offload and Attention over a given grouping."""
    rng = np.random.default_rng(13)
    cases = [(300, [64, 1, 30, 64, 41, 50, 50]), (64, [1] * 64), (128, [64, 64]), (1000, None), (77, [77 - 64, 64])]
    for n, sizes in cases:
        if sizes is None:
            order, starts = W.random_parts(rng, n, 40)
        else:
            order = rng.permutation(n).astype(np.int32)
            starts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        P = len(starts) - 1
        k, v = rand_kv(rng, n, scale=1.4)
        # index: the mean of each group's gathered rows (numpy), exact for 1-token groups
        summ = O.index_parts(k, order, starts, lib)
        kf = bf(k)
        for p in range(P):
            rows = order[starts[p]:starts[p + 1]]
            ref = kf[rows].mean(axis=0)
            assert np.abs(summ[p] - ref).max() <= 1e-12, f"group {p} mean differs"
            if len(rows) == 1:
                assert np.array_equal(summ[p], kf[rows[0]]), "a 1-token group's summary is its key"
        # offload: page p holds the group's tokens in order from row 0, then zeros
        pages = O.offload_parts(k, v, order, starts, lib)
        for p in range(P):
            rows = order[starts[p]:starts[p + 1]]
            m = len(rows)
            assert np.array_equal(pages[p, 0, :m], k[rows]) and np.array_equal(pages[p, 1, :m], v[rows])
            assert not pages[p, :, m:].any(), "page padding must be zero"
        G = 1 + n % 5
        q = f32_to_bf16_bits(rng.standard_normal((G, D)).astype(np.float32))
        # every group selected: dense attention over all tokens, whatever the grouping
        u = O.Unit.from_parts(k, v, order, starts, cap=P, lib=lib)
        r = u.step(q, k=P, t=0)
        assert list(r["sel"]) == list(range(P))
        err = np.abs(r["out"] - _sdpa(q, k, v)).max()
        assert err <= 1e-12, f"dense identity over variable partitions broken (n={n}): {err}"
        # a partial selection: the k best groups by q . mean summed over heads (numpy
        # ranking, equal scores to the lower index), then dense attention over their tokens
        kk = max(1, P // 3)
        u2 = O.Unit.from_parts(k, v, order, starts, cap=kk, lib=lib)
        r2 = u2.step(q, k=kk, t=0)
        sc = (bf(q).sum(axis=0)[None, :] * np.stack([kf[order[starts[p]:starts[p + 1]]].mean(axis=0)
                                                    for p in range(P)])).sum(axis=1)
        want = np.sort(sorted(range(P), key=lambda p: (-sc[p], p))[:kk])
        assert list(r2["sel"]) == list(want), "selection over group summaries differs from the ranking"
        rows = np.concatenate([order[starts[p]:starts[p + 1]] for p in want])
        err2 = np.abs(r2["out"] - _sdpa(q, k[rows], v[rows])).max()
        assert err2 <= 1e-12, f"partial selection must attend exactly the chosen groups' tokens: {err2}"
    # constant groups: every token of a group carries the group's key
    order, starts = W.random_parts(rng, 500, 20)
    consts = f32_to_bf16_bits(rng.standard_normal((20, D)).astype(np.float32))
    k = np.empty((500, D), np.uint16)
    for p in range(20):
        k[order[starts[p]:starts[p + 1]]] = consts[p]
    assert np.array_equal(O.index_parts(k, order, starts, lib), bf(consts)), "constant group mean"


ALL_CHECKS = [check_dense_attention, check_attention_closed_forms, check_scores_probe, check_topk_bruteforce,
              check_index, check_lru_invariants, check_lru_hand_trace, check_budget_hand_trace,
              check_step_consistency, check_append_tail, check_variable_partitions]
