"""Lockstep comparison of the CUDA path (through the C ABI) with the oracle.

Both sides take the same generator inputs; no value produced by the CUDA path
is ever fed into the oracle. Per decode step and per compared unit:

  selection   Select is stateless, so the GPU set is checked against the
              oracle's own top-k every step. The sets must be equal outside the
              tie band: partitions whose oracle score lies within 1e-5 relative
              of the k-th largest oracle score. Inside the band any choice of
              the right size is valid.
  page state  while a unit's selections have matched exactly, the oracle's
              manager has seen the same history, so slots, hits, timestamps,
              LRU cutoff and evictions, the resolved table and live segments
              must agree bit for bit. After a tie-band divergence the unit's
              state is only checked for validity (invariants below).
  outputs     max-abs error <= 2e-3 against the oracle's attention over the
              oracle-enumerated valid set equal to the GPU's set (the oracle's
              own set when nothing diverged).

Validity invariants checked for every unit of every exported layer: slots hold
distinct partitions, resolve(p) = s iff slot s holds p, live segments equal the
occupied 64-partition ranges, the selection is ascending and resident in the
slots it names, those slots carry the current step.

KV append (tail mode, ``append > 0``): each step first appends the request's next
token (drawn by the generator beyond the initial context) on both sides, then
decodes. The oracle's TailUnit supplies the expected partitions and tail; the
compared units' tail pages must equal the oracle's tail byte for byte and the
summaries of partitions made from full tails must match the oracle's means.

Variable partitions (workloads with ``mean_part > 0``): both sides take the
generator's grouping (token order and partition boundaries); the GPU's summaries
must match the oracle's group means and, on the first step, every resident page
must equal the oracle's page of its partition byte for byte.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field
from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np

import oracle as O
import workload as W

OUT_TOL = 2e-3
TIE_REL = 1e-5


@dataclass
class Report:
    steps: int = 0
    compared_units: int = 0
    exact_units: int = 0
    tie_divergences: int = 0
    max_out_err: float = 0.0
    evictions: int = 0
    misses: int = 0
    hits: int = 0
    notes: List[str] = field(default_factory=list)


def tie_band(sc: np.ndarray, keff: int) -> Tuple[np.ndarray, float]:
    order = np.lexsort((np.arange(sc.size), -sc))
    kth = sc[order[keff - 1]]
    band = np.abs(sc - kth) <= TIE_REL * abs(kth)
    return band, kth


def check_selection(sc: np.ndarray, sel_o: np.ndarray, sel_g: np.ndarray, where: str) -> bool:
    """True when identical; False when different only inside the tie band; raises otherwise."""
    if np.array_equal(sel_o, sel_g):
        return True
    keff = sel_o.size
    assert sel_g.size == keff, f"{where}: GPU selected {sel_g.size} partitions, oracle {keff}"
    assert np.all(np.diff(sel_g) > 0), f"{where}: GPU selection not strictly ascending"
    band, kth = tie_band(sc, keff)
    so, sg = set(sel_o.tolist()), set(sel_g.tolist())
    outside_o = {p for p in so if not band[p]}
    outside_g = {p for p in sg if not band[p]}
    assert outside_o == outside_g, (
        f"{where}: selections differ outside the tie band: oracle-only {sorted(so - sg)}, gpu-only {sorted(sg - so)}, "
        f"k-th score {kth!r}, scores {[float(sc[p]) for p in sorted(so ^ sg)]}")
    return False


def valid_sets(sc: np.ndarray, sel_o: np.ndarray) -> Iterable[np.ndarray]:
    """All selections the tie band allows (oracle arithmetic only)."""
    keff = sel_o.size
    band, _ = tie_band(sc, keff)
    fixed = [p for p in sel_o.tolist() if not band[p]]
    cands = np.nonzero(band)[0].tolist()
    need = keff - len(fixed)
    for comb in itertools.combinations(cands, need):
        yield np.array(sorted(fixed + list(comb)), np.int32)


def check_invariants(ex: dict, ul: int, P: int, t: int, where: str):
    sp = ex["slot_part"][ul]
    lu = ex["last_use"][ul]
    res = [int(p) for p in sp if p >= 0]
    assert len(set(res)) == len(res), f"{where}: a partition is resident twice"
    assert all(0 <= p < P for p in res), f"{where}: resident partition out of range"
    if "resolve" in ex:
        rs = ex["resolve"][ul][:P]
        for p in range(P):
            s = rs[p]
            if s >= 0:
                assert sp[s] == p, f"{where}: resolve({p}) = {s} but slot holds {sp[s]}"
        assert sum(1 for p in range(P) if rs[p] >= 0) == len(res), f"{where}: resolve misses resident pages"
        assert ex["live_segs"][ul] == len({p // 64 for p in res}), f"{where}: live segments mismatch"
    keff = int(ex["keff"][ul])
    sel = ex["sel"][ul][:keff]
    assert np.all(np.diff(sel) > 0), f"{where}: selection not ascending"
    for p, s in zip(sel, ex["sel_slot"][ul][:keff]):
        assert sp[s] == p, f"{where}: selected partition {p} not in its slot {s}"
        assert lu[s] == t, f"{where}: selected slot {s} has last_use {lu[s]} at step {t}"


class Lockstep:
    """Runs a workload on the GPU and the oracle side by side on chosen units."""

    def __init__(self, w: W.Workload, units: Optional[List[Tuple[int, int, int]]] = None, device: int = 0,
                 flags: int = 0, seg_pool_segments: int = 0, offload_from_device: bool = False,
                 gen_threads: int = 0, append: int = 0, budgets=None):
        import torch
        from sparse_attention_tiered_gb300 import SpinContext
        self.torch = torch
        self.w = w
        self.append = append
        self.budgets = budgets or {}  # step -> [(request, pages)]: buffer elasticity events
        self.budget_b = [w.cap] * w.B
        self.dev = torch.device(f"cuda:{device}")
        self.units = units if units is not None else [(l, b, h) for l in range(w.L) for b in range(w.B)
                                                      for h in range(w.Hkv)]
        self.ctx = SpinContext.for_workload(w, device=device, flags=flags, seg_pool_segments=seg_pool_segments,
                                            append_tokens=append)
        self.oracle: Dict[Tuple[int, int, int], O.Unit] = {}
        self.fresh_cap = max(w.topk, 1)
        # tail mode: the generator draws each request's tokens past the initial context too;
        # those are the appended tokens, [L][B] -> [Hkv][append][128]
        wf = w.with_(ctx_len=[n + append for n in w.ctx_len]) if append else w
        self.new_kv = {}
        want = {}
        for (l, b, h) in self.units:
            want.setdefault((l, b), []).append(h)
        self.parts = bool(getattr(w, "mean_part", 0))
        for l in range(w.L):
            for b in range(w.B):
                n = w.ctx_len[b]
                k, v = wf.request_kv(l, b, threads=gen_threads)
                if self.parts:
                    order, starts = w.request_parts(l, b)
                if append:
                    self.new_kv[(l, b)] = (np.ascontiguousarray(k[:, n:]), np.ascontiguousarray(v[:, n:]))
                    k, v = np.ascontiguousarray(k[:, :n]), np.ascontiguousarray(v[:, :n])
                if offload_from_device:
                    kd = torch.from_numpy(k.view(np.int16)).to(self.dev)
                    vd = torch.from_numpy(v.view(np.int16)).to(self.dev)
                    if self.parts:
                        self.ctx.index_offload_parts(b, l, kd, vd, order, starts)
                    else:
                        self.ctx.index_offload_device(b, l, kd, vd)
                    torch.cuda.synchronize()
                    del kd, vd
                elif self.parts:
                    self.ctx.index_offload_parts(b, l, k, v, order, starts)
                else:
                    self.ctx.index_offload_host(b, l, k, v)
                    torch.cuda.synchronize()  # the host arrays are reused/freed next
                for h in want.get((l, b), []):
                    if self.parts:
                        self.oracle[(l, b, h)] = O.Unit.from_parts(np.ascontiguousarray(k[h]),
                                                                   np.ascontiguousarray(v[h]), order[h], starts[h],
                                                                   w.cap)
                    elif append:
                        self.oracle[(l, b, h)] = O.TailUnit(np.ascontiguousarray(k[h]), np.ascontiguousarray(v[h]),
                                                            w.cap, append)
                    else:
                        self.oracle[(l, b, h)] = O.Unit(n, w.cap, np.ascontiguousarray(k[h]),
                                                        np.ascontiguousarray(v[h]))
        self.diverged = set()
        self.qs = w.queries()
        self.t = 0
        self.out = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32, device=self.dev)
        self.report = Report()

    def close(self):
        self.ctx.close()

    def step(self, check: bool = True):
        torch = self.torch
        w = self.w
        qb = self.qs.bf16()
        qd = torch.from_numpy(qb.view(np.int16)).to(self.dev)
        for (b, pages) in self.budgets.get(self.t, []):
            self.ctx.set_buffer(b, pages)
            self.budget_b[b] = pages
            for (l, bb, h), u in self.oracle.items():
                if bb == b:
                    u.set_budget(pages)
        if self.append:
            t = self.t
            for l in range(w.L):
                kn = np.stack([self.new_kv[(l, b)][0][:, t] for b in range(w.B)])  # [B][Hkv][128]
                vn = np.stack([self.new_kv[(l, b)][1][:, t] for b in range(w.B)])
                kd = torch.from_numpy(kn.view(np.int16)).to(self.dev)
                vd = torch.from_numpy(vn.view(np.int16)).to(self.dev)
                self.ctx.append_kv(l, kd, vd)
                for (ll, b, h), u in self.oracle.items():
                    if ll == l:
                        u.append(kn[b, h], vn[b, h])
        for l in range(w.L):
            self.ctx.decode_step(l, qd[l], self.out[l])
        torch.cuda.synchronize()
        if check:
            self._check(qb)
        self.qs.advance()
        self.t += 1
        self.report.steps += 1

    def _check(self, qb: np.ndarray):
        w, t = self.w, self.t
        out = self.out.cpu().numpy()
        layers = sorted({l for (l, _, _) in self.units})
        exports = {l: self.ctx.export(l, resolve=True) for l in layers}
        rep = self.report
        for l in layers:
            ex = exports[l]
            for b in range(w.B):
                for h in range(w.Hkv):
                    check_invariants(ex, b * w.Hkv + h, self.ctx.P_lb[l][b], t, f"step {t} unit {(l, b, h)}")
                    resident = int((ex["slot_part"][b * w.Hkv + h] >= 0).sum())
                    assert resident <= self.budget_b[b], (
                        f"step {t} unit {(l, b, h)}: {resident} pages resident over the budget {self.budget_b[b]}")
        for (l, b, h), u in self.oracle.items():
            ex = exports[l]
            ul = b * w.Hkv + h
            where = f"step {t} unit {(l, b, h)}"
            q = np.ascontiguousarray(qb[l, b, h * w.G:(h + 1) * w.G])
            g_out = out[l, b, h * w.G:(h + 1) * w.G]
            rep.compared_units += 1
            if self.append:
                assert u.P == self.ctx.P_lb[l][b], f"{where}: partition count differs"
                tail = self.ctx.read_tail(l, b, h)
                assert np.array_equal(tail[:, :u.tail_n], u.tail[:, :u.tail_n]), f"{where}: tail page differs"
                assert not tail[:, u.tail_n:].any(), f"{where}: tail page not clear past its tokens"
                if u.P:
                    gs = self.ctx.summaries(l, b, h).astype(np.float64)
                    serr = float(np.abs(gs - u.summ).max())
                    assert serr <= 1e-5, f"{where}: summaries differ by {serr}"
            if self.parts:
                # variable partitions: the GPU's Index over the same grouping, and (first step)
                # every resident page byte for byte against the oracle's page of that partition
                assert u.P == self.ctx.P_lb[l][b], f"{where}: partition count differs"
                if u.P:
                    gs = self.ctx.summaries(l, b, h).astype(np.float64)
                    serr = float(np.abs(gs - u.summ).max())
                    assert serr <= 1e-5, f"{where}: summaries differ by {serr}"
                if t == 0:
                    for s_, p_ in enumerate(ex["slot_part"][ul]):
                        if p_ >= 0:
                            pg = self.ctx.read_page(l, b, h, s_)
                            assert np.array_equal(pg, u.host_pages[p_]), f"{where}: page of partition {p_} differs"
            if u.P == 0 and not (self.append and u.tail_n):
                assert np.all(g_out == 0), f"{where}: empty request must give zeros"
                continue
            sc = O.scores(u.summ, q)
            sel_o = O.topk(sc, w.topk)
            keff = int(ex["keff"][ul])
            sel_g = ex["sel"][ul][:keff].copy()
            same = check_selection(sc, sel_o, sel_g, where)
            key = (l, b, h)
            if same and key not in self.diverged:
                ss, hit, vic, mo = u.manage(sel_o, t)
                o_out = u.attend(sel_o, ss, q)
                assert mo.error == 0, f"{where}: oracle page pool error"
                info = ex["unit_info"][ul]
                assert np.array_equal(ex["sel_slot"][ul][:keff], ss), f"{where}: slots differ"
                assert np.array_equal(ex["sel_hit"][ul][:keff].astype(bool), hit), f"{where}: hits differ"
                assert (info[0], info[1], info[2], info[3], info[4], info[5]) == (
                    mo.hits, mo.misses, mo.resident_before, mo.demand, mo.cutoff, mo.evicted), (
                    f"{where}: manager record differs: gpu {info[:6].tolist()} oracle "
                    f"{[mo.hits, mo.misses, mo.resident_before, mo.demand, mo.cutoff, mo.evicted]}")
                sp, lu, rs = u.export()
                assert np.array_equal(ex["slot_part"][ul], sp), f"{where}: slot map differs"
                assert np.array_equal(ex["last_use"][ul], lu), f"{where}: timestamps differ"
                assert np.array_equal(ex["resolve"][ul][:u.P], rs), f"{where}: page table differs"
                assert ex["live_segs"][ul] == u.live_segments(), f"{where}: live segments differ"
                rep.exact_units += 1
                rep.evictions += mo.evicted
                rep.misses += mo.misses
                rep.hits += mo.hits
            else:
                if key not in self.diverged:
                    self.diverged.add(key)
                    rep.tie_divergences += 1
                    rep.notes.append(f"{where}: tie-band divergence")
                match = None
                for cand in valid_sets(sc, sel_o):
                    if np.array_equal(cand, sel_g):
                        match = cand
                        break
                assert match is not None, f"{where}: GPU set is not one of the valid tie-band sets"
                fresh = u.clone_empty(self.fresh_cap)
                ss, _, _, _ = fresh.manage(match, 0)
                o_out = fresh.attend(match, ss, q)
            err = float(np.abs(g_out - o_out).max())
            rep.max_out_err = max(rep.max_out_err, err)
            assert err <= OUT_TOL, f"{where}: output max-abs error {err} > {OUT_TOL}"


def sample_units(w: W.Workload, n: int, seed: int = 0) -> List[Tuple[int, int, int]]:
    rng = np.random.default_rng(seed)
    allu = [(l, b, h) for l in range(w.L) for b in range(w.B) for h in range(w.Hkv)]
    idx = rng.choice(len(allu), size=min(n, len(allu)), replace=False)
    return sorted(allu[i] for i in idx)


class AllUnits:
    """Every unit of a fixed-partition workload, GPU against the oracle every step.

    The oracle side runs all units of a step with its thread pool (step_units_full).
    Per step and layer: selections are checked against the oracle's top-k with the
    tie band; for every unit whose selections have always matched exactly, slots,
    hits, the manager record, slot map, timestamps, the resolved two-level table and
    live segments are compared bit for bit (vectorised over the layer) and outputs
    within OUT_TOL. A unit that diverged inside the tie band is checked for validity
    (invariants) and its output against the oracle's attention over the GPU's set.
    """

    def __init__(self, w: W.Workload, device: int = 0, flags: int = 0, gen_threads: int = 0, threads: int = 0):
        import torch
        from sparse_attention_tiered_gb300 import SpinContext
        assert not getattr(w, "mean_part", 0), "fixed partitions only"
        self.torch = torch
        self.w = w
        self.threads = threads
        self.dev = torch.device(f"cuda:{device}")
        self.ctx = SpinContext.for_workload(w, device=device, flags=flags)
        self.units: List[O.Unit] = []
        self.keys: List[Tuple[int, int, int]] = []
        for l in range(w.L):
            for b in range(w.B):
                k, v = w.request_kv(l, b, threads=gen_threads)
                self.ctx.index_offload_host(b, l, k, v)
                torch.cuda.synchronize()  # the host arrays are reused/freed next
                for h in range(w.Hkv):
                    self.units.append(O.Unit(w.ctx_len[b], w.cap, np.ascontiguousarray(k[h]),
                                             np.ascontiguousarray(v[h])))
                    self.keys.append((l, b, h))
                del k, v
        self.Ul = w.B * w.Hkv
        self.diverged = np.zeros(len(self.units), bool)
        self.qs = w.queries()
        self.t = 0
        self.out = torch.empty((w.L, w.B, w.Hq, 128), dtype=torch.float32, device=self.dev)
        self.report = Report()
        self.exact_unit_steps = 0

    def close(self):
        self.ctx.close()
        self.units = []

    def step(self):
        torch, w, t = self.torch, self.w, self.t
        qb = self.qs.bf16()
        qd = torch.from_numpy(qb.view(np.int16)).to(self.dev)
        for l in range(w.L):
            self.ctx.decode_step(l, qd[l], self.out[l])
        qlist = [np.ascontiguousarray(qb[l, b, h * w.G:(h + 1) * w.G]) for (l, b, h) in self.keys]
        res = O.step_units_full(self.units, qlist, w.topk, t, threads=self.threads)
        torch.cuda.synchronize()
        out = self.out.cpu().numpy()
        for l in range(w.L):
            self._check_layer(l, qb, out, res[l * self.Ul:(l + 1) * self.Ul])
        self.report.steps += 1
        self.qs.advance()
        self.t += 1

    def _check_layer(self, l, qb, out, res):
        w, t, rep = self.w, self.t, self.report
        ex = self.ctx.export(l, resolve=True)
        U, cap, Pm = self.Ul, w.cap, self.ctx.P_max
        base = l * U
        sp_o = np.empty((U, cap), np.int32)
        lu_o = np.empty((U, cap), np.int32)
        rs_o = np.full((U, max(Pm, 1)), -1, np.int32)
        live_o = np.empty(U, np.int32)
        out_o = np.empty((U, w.G, 128), np.float64)
        exact = np.zeros(U, bool)
        for ul in range(U):
            i = base + ul
            u, r = self.units[i], res[ul]
            b, h = ul // w.Hkv, ul % w.Hkv
            where = f"step {t} unit {(l, b, h)}"
            rep.compared_units += 1
            keff = int(ex["keff"][ul])
            sel_g = ex["sel"][ul][:keff]
            if u.P == 0:
                assert keff == 0 and np.all(out[l, b, h * w.G:(h + 1) * w.G] == 0), f"{where}: empty request"
                exact[ul] = not self.diverged[i]
                sp_o[ul], lu_o[ul], _ = u.export()
                live_o[ul] = u.live_segments()
                out_o[ul] = 0.0
                continue
            same = check_selection(r["scores"], r["sel"], sel_g, where)
            if same and not self.diverged[i]:
                exact[ul] = True
                sp, lu, rs = u.export()
                sp_o[ul], lu_o[ul] = sp, lu
                rs_o[ul, :u.P] = rs
                live_o[ul] = u.live_segments()
                out_o[ul] = r["out"]
                mo = r["mo"]
                assert r["mo"].error == 0, f"{where}: oracle page pool error"
                info = ex["unit_info"][ul]
                if (info[0], info[1], info[2], info[3], info[4], info[5]) != (
                        mo.hits, mo.misses, mo.resident_before, mo.demand, mo.cutoff, mo.evicted):
                    raise AssertionError(f"{where}: manager record differs: gpu {info[:6].tolist()} oracle "
                                         f"{[mo.hits, mo.misses, mo.resident_before, mo.demand, mo.cutoff, mo.evicted]}")
                assert np.array_equal(ex["sel_slot"][ul][:keff], r["sel_slot"]), f"{where}: slots differ"
                assert np.array_equal(ex["sel_hit"][ul][:keff].astype(bool), r["sel_hit"]), f"{where}: hits differ"
                rep.evictions += mo.evicted
                rep.misses += mo.misses
                rep.hits += mo.hits
            else:
                if not self.diverged[i]:
                    self.diverged[i] = True
                    rep.tie_divergences += 1
                    rep.notes.append(f"{where}: tie-band divergence")
                check_invariants(ex, ul, u.P, t, where)
                match = None
                for cand in valid_sets(r["scores"], r["sel"]):
                    if np.array_equal(cand, sel_g):
                        match = cand
                        break
                assert match is not None, f"{where}: GPU set is not one of the valid tie-band sets"
                fresh = u.clone_empty(max(w.topk, 1))
                ss, _, _, _ = fresh.manage(match, 0)
                q = np.ascontiguousarray(qb[l, b, h * w.G:(h + 1) * w.G])
                o_div = fresh.attend(match, ss, q)
                err = float(np.abs(out[l, b, h * w.G:(h + 1) * w.G] - o_div).max())
                rep.max_out_err = max(rep.max_out_err, err)
                assert err <= OUT_TOL, f"{where}: output max-abs error {err} > {OUT_TOL}"
        # bit-exact page state and outputs of every exact unit, vectorised over the layer
        idx = np.nonzero(exact)[0]
        self.exact_unit_steps += len(idx)
        rep.exact_units += len(idx)
        if len(idx):
            for name, g_arr, o_arr in (("slot map", ex["slot_part"], sp_o), ("timestamps", ex["last_use"], lu_o),
                                       ("page table", ex["resolve"][:, :max(Pm, 1)], rs_o),
                                       ("live segments", ex["live_segs"], live_o)):
                bad = np.nonzero(np.any((g_arr[idx] != o_arr[idx]).reshape(len(idx), -1), axis=1))[0]
                if len(bad):
                    ul = int(idx[bad[0]])
                    raise AssertionError(f"step {t} unit {(l, ul // w.Hkv, ul % w.Hkv)}: {name} differs")
            g_out = out[l].reshape(w.B, w.Hkv, w.G, 128).reshape(U, w.G, 128)
            err = float(np.abs(g_out[idx] - out_o[idx]).max())
            rep.max_out_err = max(rep.max_out_err, err)
            assert err <= OUT_TOL, f"step {t} layer {l}: output max-abs error {err} > {OUT_TOL}"
