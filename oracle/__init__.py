"""Python access to the SPIN decode-step oracle (``spin_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``. The product path never loads it.

The oracle shares no code with the CUDA library; both take their inputs from
the ``workload`` generator. See ``spin_oracle.c`` for the page citations and
the readings taken where the pages leave a rule open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D = 128
PART = 64
PAGE_ELEMS = 2 * PART * D


def build(force: bool = False, out: Optional[str] = None, defines=()) -> str:
    """Compile spin_oracle.c into a shared library (gcc, OpenMP when available)."""
    src = os.path.join(_HERE, "spin_oracle.c")
    dst = out or _LIB_PATH
    if not force and out is None and os.path.exists(dst) and os.path.getmtime(dst) >= os.path.getmtime(src):
        return dst
    extra = [f"-D{d}" for d in defines]
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11"] + extra + [src, "-o", dst + ".tmp",
                                                                                             "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(dst + ".tmp", dst)
    return dst


class ManageOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hits", "misses", "resident_before", "free_before", "demand", "cutoff", "evicted", "error")]


class StepIO(ctypes.Structure):
    _fields_ = [
        ("summ", ctypes.c_void_p),
        ("host_pages", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("G", ctypes.c_int32),
        ("k", ctypes.c_int32),
        ("t", ctypes.c_int32),
        ("scores", ctypes.c_void_p),
        ("sel", ctypes.c_void_p),
        ("sel_slot", ctypes.c_void_p),
        ("sel_hit", ctypes.c_void_p),
        ("victims", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("mo", ManageOut),
        ("keff", ctypes.c_int32),
    ]


def _bind(L):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.oracle_index.argtypes = [vp, i64, vp]
    L.oracle_offload.argtypes = [vp, vp, i64, vp]
    L.oracle_scores.argtypes = [vp, i64, vp, i32, vp]
    L.oracle_topk.argtypes = [vp, i64, i32, vp]
    L.oracle_topk.restype = i32
    L.oracle_unit_create.argtypes = [i32, i32]
    L.oracle_unit_create.restype = vp
    L.oracle_unit_destroy.argtypes = [vp]
    L.oracle_resolve.argtypes = [vp, i32]
    L.oracle_resolve.restype = i32
    L.oracle_live_segments.argtypes = [vp]
    L.oracle_live_segments.restype = i32
    L.oracle_manage.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, ctypes.POINTER(ManageOut)]
    L.oracle_attend.argtypes = [vp, vp, vp, i32, vp, i32, vp]
    L.oracle_step_unit.argtypes = [vp, ctypes.POINTER(StepIO)]
    L.oracle_step_units.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(StepIO), i32, i32]
    L.oracle_step_units.restype = i32
    L.oracle_unit_export.argtypes = [vp, vp, vp, vp]
    L.oracle_unit_slot.argtypes = [vp, i32]
    L.oracle_unit_slot.restype = vp
    L.oracle_unit_create_tail.argtypes = [i32, i32, i32]
    L.oracle_unit_create_tail.restype = vp
    L.oracle_unit_grow.argtypes = [vp]
    L.oracle_unit_set_budget.argtypes = [vp, i32]
    L.oracle_unit_set_budget.restype = i32
    L.oracle_unit_grow.restype = i32
    L.oracle_attend_tail.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, vp]
    L.oracle_index_parts.argtypes = [vp, vp, vp, i32, vp]
    L.oracle_offload_parts.argtypes = [vp, vp, vp, vp, i32, vp]
    L.oracle_unit_create_parts.argtypes = [vp, i32, i32]
    L.oracle_unit_create_parts.restype = vp
    return L


def load(path: Optional[str] = None):
    """The oracle library (built on first use). `path` loads another build (mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------------------
# Stateless pieces
# ---------------------------------------------------------------------------

def index(k_bits: np.ndarray, lib=None) -> np.ndarray:
    """Partition mean keys, double [P][128], from bf16 bits K [ntok][128]."""
    lib = lib or load()
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    n = k_bits.shape[0]
    P = (n + PART - 1) // PART
    s = np.empty((P, D), np.float64)
    lib.oracle_index(_p(k_bits), n, _p(s))
    return s


def offload(k_bits: np.ndarray, v_bits: np.ndarray, lib=None) -> np.ndarray:
    """Host pages [P][2][64][128] bf16 bits (zero padded)."""
    lib = lib or load()
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    n = k_bits.shape[0]
    P = (n + PART - 1) // PART
    pages = np.empty((P, 2, PART, D), np.uint16)
    lib.oracle_offload(_p(k_bits), _p(v_bits), n, _p(pages))
    return pages


def _parts_args(order: np.ndarray, starts: np.ndarray):
    order = np.ascontiguousarray(order, np.int32)
    starts = np.ascontiguousarray(starts, np.int32)
    return order, starts, starts.shape[0] - 1


def index_parts(k_bits: np.ndarray, order: np.ndarray, starts: np.ndarray, lib=None) -> np.ndarray:
    """Mean keys, double [P][128], of variable partitions: partition p holds the tokens
    order[starts[p]:starts[p+1]] of K [ntok][128] (bf16 bits)."""
    lib = lib or load()
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    order, starts, P = _parts_args(order, starts)
    s = np.empty((max(P, 1), D), np.float64)
    lib.oracle_index_parts(_p(k_bits), _p(order), _p(starts), P, _p(s))
    return s[:P]


def offload_parts(k_bits: np.ndarray, v_bits: np.ndarray, order: np.ndarray, starts: np.ndarray,
                  lib=None) -> np.ndarray:
    """Host pages [P][2][64][128] of variable partitions: page p holds its partition's
    tokens in order from row 0, zero padded."""
    lib = lib or load()
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    order, starts, P = _parts_args(order, starts)
    pages = np.empty((max(P, 1), 2, PART, D), np.uint16)
    lib.oracle_offload_parts(_p(k_bits), _p(v_bits), _p(order), _p(starts), P, _p(pages))
    return pages[:P]


def scores(summ: np.ndarray, q_bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    summ = np.ascontiguousarray(summ, np.float64)
    q_bits = np.ascontiguousarray(q_bits, np.uint16)
    sc = np.empty(summ.shape[0], np.float64)
    lib.oracle_scores(_p(summ), summ.shape[0], _p(q_bits), q_bits.shape[0], _p(sc))
    return sc


def topk(sc: np.ndarray, k: int, lib=None) -> np.ndarray:
    lib = lib or load()
    sc = np.ascontiguousarray(sc, np.float64)
    sel = np.empty(max(k, 1), np.int32)
    keff = lib.oracle_topk(_p(sc), sc.shape[0], k, _p(sel))
    return sel[:keff].copy()


# ---------------------------------------------------------------------------
# Stateful unit
# ---------------------------------------------------------------------------

class Unit:
    """Oracle page state of one (request, layer, KV head) unit."""

    def __init__(self, ntok: int, cap: int, k_bits: Optional[np.ndarray] = None,
                 v_bits: Optional[np.ndarray] = None, lib=None):
        self.lib = lib or load()
        self.ntok = ntok
        self.cap = cap
        self.P = (ntok + PART - 1) // PART
        self.h = self.lib.oracle_unit_create(ntok, cap)
        self.summ = None
        self.host_pages = None
        self.part_n = None
        if k_bits is not None:
            self.load_kv(k_bits, v_bits)

    @classmethod
    def from_parts(cls, k_bits: np.ndarray, v_bits: np.ndarray, order: np.ndarray, starts: np.ndarray, cap: int,
                   lib=None) -> "Unit":
        """Unit of variable partitions (Index and Offload over the given grouping)."""
        u = cls.__new__(cls)
        u.lib = lib or load()
        starts = np.ascontiguousarray(starts, np.int32)
        u.part_n = np.ascontiguousarray(np.diff(starts), np.int32)
        u.P = int(u.part_n.shape[0])
        u.ntok = int(starts[-1])
        u.cap = cap
        u.h = u.lib.oracle_unit_create_parts(_p(u.part_n) if u.P else None, u.P, cap)
        u.summ = index_parts(k_bits, order, starts, u.lib)
        u.host_pages = offload_parts(k_bits, v_bits, order, starts, u.lib)
        return u

    def clone_empty(self, cap: int) -> "Unit":
        """A unit with the same partitions, summaries and host pages, and nothing resident."""
        c = Unit.__new__(Unit)
        c.lib, c.cap, c.ntok, c.P, c.part_n = self.lib, cap, self.ntok, self.P, self.part_n
        if self.part_n is not None:
            c.h = self.lib.oracle_unit_create_parts(_p(self.part_n) if self.P else None, self.P, cap)
        else:
            c.h = self.lib.oracle_unit_create(self.ntok, cap)
        c.summ, c.host_pages = self.summ, self.host_pages
        return c

    def load_kv(self, k_bits: np.ndarray, v_bits: np.ndarray):
        """Index + Offload of this unit's keys and values."""
        assert k_bits.shape[0] == self.ntok
        self.summ = index(k_bits, self.lib)
        self.host_pages = offload(k_bits, v_bits, self.lib)

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.oracle_unit_destroy(h)
            self.h = None

    def resolve(self, p: int) -> int:
        return self.lib.oracle_resolve(self.h, p)

    def set_budget(self, pages: int):
        """Buffer elasticity: the unit may keep at most `pages` resident from the next step on."""
        assert self.lib.oracle_unit_set_budget(self.h, pages) == 0, "budget outside [1, cap]"

    def live_segments(self) -> int:
        return self.lib.oracle_live_segments(self.h)

    def export(self):
        sp = np.empty(self.cap, np.int32)
        lu = np.empty(self.cap, np.int32)
        rs = np.empty(max(self.P, 1), np.int32)
        self.lib.oracle_unit_export(self.h, _p(sp), _p(lu), _p(rs))
        return sp, lu, rs[:self.P]

    def slot_page(self, s: int) -> np.ndarray:
        ptr = self.lib.oracle_unit_slot(self.h, s)
        buf = (ctypes.c_uint16 * PAGE_ELEMS).from_address(ptr)
        return np.frombuffer(buf, np.uint16).copy().reshape(2, PART, D)

    def manage(self, sel: np.ndarray, t: int):
        sel = np.ascontiguousarray(sel, np.int32)
        k = sel.shape[0]
        sel_slot = np.empty(max(k, 1), np.int32)
        sel_hit = np.empty(max(k, 1), np.uint8)
        victims = np.empty(self.cap, np.int32)
        mo = ManageOut()
        self.lib.oracle_manage(self.h, _p(sel), k, t, _p(self.host_pages), _p(sel_slot), _p(sel_hit), _p(victims),
                               ctypes.byref(mo))
        return sel_slot[:k].copy(), sel_hit[:k].astype(bool), victims[:mo.evicted].copy(), mo

    def attend(self, sel: np.ndarray, sel_slot: np.ndarray, q_bits: np.ndarray) -> np.ndarray:
        sel = np.ascontiguousarray(sel, np.int32)
        sel_slot = np.ascontiguousarray(sel_slot, np.int32)
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        G = q_bits.shape[0]
        out = np.empty((G, D), np.float64)
        self.lib.oracle_attend(self.h, _p(sel), _p(sel_slot), sel.shape[0], _p(q_bits), G, _p(out))
        return out

    def step(self, q_bits: np.ndarray, k: int, t: int) -> dict:
        """Select -> Manage/Retrieve -> Attention for one decode step."""
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        G = q_bits.shape[0]
        sc = np.empty(max(self.P, 1), np.float64)
        sel = np.empty(max(k, 1), np.int32)
        sel_slot = np.empty(max(k, 1), np.int32)
        sel_hit = np.empty(max(k, 1), np.uint8)
        victims = np.empty(self.cap, np.int32)
        out = np.empty((G, D), np.float64)
        io = StepIO(self.summ.ctypes.data, self.host_pages.ctypes.data, q_bits.ctypes.data, G, k, t,
                    sc.ctypes.data, sel.ctypes.data, sel_slot.ctypes.data, sel_hit.ctypes.data,
                    victims.ctypes.data, out.ctypes.data)
        self.lib.oracle_step_unit(self.h, ctypes.byref(io))
        keff = io.keff
        return dict(scores=sc[:self.P].copy(), sel=sel[:keff].copy(), sel_slot=sel_slot[:keff].copy(),
                    sel_hit=sel_hit[:keff].astype(bool), victims=victims[:io.mo.evicted].copy(), out=out,
                    mo=io.mo)


def step_units_parallel(units, qs, k: int, t: int, threads: int = 0, lib=None):
    """Run one decode step on many units with the oracle's thread pool; returns threads used."""
    lib = lib or load()
    n = len(units)
    handles = (ctypes.c_void_p * n)(*[u.h for u in units])
    ios = (StepIO * n)()
    keep = []
    for i, (u, q) in enumerate(zip(units, qs)):
        q = np.ascontiguousarray(q, np.uint16)
        sel = np.empty(max(k, 1), np.int32)
        ss = np.empty(max(k, 1), np.int32)
        sh = np.empty(max(k, 1), np.uint8)
        out = np.empty((q.shape[0], D), np.float64)
        keep.append((q, sel, ss, sh, out))
        ios[i] = StepIO(u.summ.ctypes.data, u.host_pages.ctypes.data, q.ctypes.data, q.shape[0], k, t, None,
                        sel.ctypes.data, ss.ctypes.data, sh.ctypes.data, None, out.ctypes.data)
    used = lib.oracle_step_units(handles, ios, n, threads)
    return used, keep


def step_units_full(units, qs, k: int, t: int, threads: int = 0, lib=None):
    """One decode step on many units with the oracle's thread pool, keeping every output:
    a list of dicts (scores, sel, sel_slot, sel_hit, out, mo) in the order of `units`."""
    lib = lib or load()
    n = len(units)
    handles = (ctypes.c_void_p * n)(*[u.h for u in units])
    ios = (StepIO * n)()
    keep = []
    for i, (u, q) in enumerate(zip(units, qs)):
        q = np.ascontiguousarray(q, np.uint16)
        sc = np.empty(max(u.P, 1), np.float64)
        sel = np.empty(max(k, 1), np.int32)
        ss = np.empty(max(k, 1), np.int32)
        sh = np.empty(max(k, 1), np.uint8)
        out = np.empty((q.shape[0], D), np.float64)
        keep.append((q, sc, sel, ss, sh, out))
        ios[i] = StepIO(u.summ.ctypes.data, u.host_pages.ctypes.data, q.ctypes.data, q.shape[0], k, t, sc.ctypes.data,
                        sel.ctypes.data, ss.ctypes.data, sh.ctypes.data, None, out.ctypes.data)
    lib.oracle_step_units(handles, ios, n, threads)
    res = []
    for i, (u, (q, sc, sel, ss, sh, out)) in enumerate(zip(units, keep)):
        keff = ios[i].keff
        res.append(dict(scores=sc[:u.P], sel=sel[:keff].copy(), sel_slot=ss[:keff].copy(),
                        sel_hit=sh[:keff].astype(bool), out=out, mo=ios[i].mo))
    return res


class TailUnit:
    """Oracle unit with KV append: complete 64-token partitions are selectable; the tail
    (fewer than 64 newest tokens) is attended at every step and becomes a partition
    (summarised and offloaded) when it fills."""

    def __init__(self, k_bits: np.ndarray, v_bits: np.ndarray, cap: int, append_max: int, lib=None):
        self.lib = lib or load()
        n = k_bits.shape[0]
        self.cap = cap
        self.ntok = n
        Pc = n // PART
        P_cap = (n + append_max + PART - 1) // PART
        self.P_cap = P_cap
        self.h = self.lib.oracle_unit_create_tail(Pc, max(P_cap, 1), cap)
        self.summ = index(k_bits[:Pc * PART], self.lib) if Pc else np.zeros((0, D))
        self.host_pages = offload(k_bits[:Pc * PART], v_bits[:Pc * PART], self.lib) if Pc else \
            np.zeros((0, 2, PART, D), np.uint16)
        self.tail = np.zeros((2, PART, D), np.uint16)
        self.tail_n = n - Pc * PART
        self.tail[0, :self.tail_n] = k_bits[Pc * PART:]
        self.tail[1, :self.tail_n] = v_bits[Pc * PART:]

    @property
    def P(self) -> int:
        return self.summ.shape[0]

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.oracle_unit_destroy(h)
            self.h = None

    def append(self, k_row: np.ndarray, v_row: np.ndarray):
        """One new token (bf16 bits [128] each)."""
        self.tail[0, self.tail_n] = k_row
        self.tail[1, self.tail_n] = v_row
        self.tail_n += 1
        self.ntok += 1
        if self.tail_n == PART:
            self.summ = np.concatenate([self.summ, index(self.tail[0], self.lib)])
            self.host_pages = np.concatenate([self.host_pages, self.tail[None].copy()])
            assert self.lib.oracle_unit_grow(self.h) == 0, "append beyond the unit's capacity"
            self.tail_n = 0

    def export(self):
        sp = np.empty(self.cap, np.int32)
        lu = np.empty(self.cap, np.int32)
        rs = np.empty(max(self.P_cap, 1), np.int32)
        self.lib.oracle_unit_export(self.h, _p(sp), _p(lu), _p(rs))
        return sp, lu, rs[:self.P]

    def live_segments(self) -> int:
        return self.lib.oracle_live_segments(self.h)

    def set_budget(self, pages: int):
        assert self.lib.oracle_unit_set_budget(self.h, pages) == 0, "budget outside [1, cap]"

    def manage(self, sel: np.ndarray, t: int):
        sel = np.ascontiguousarray(sel, np.int32)
        k = sel.shape[0]
        sel_slot = np.empty(max(k, 1), np.int32)
        sel_hit = np.empty(max(k, 1), np.uint8)
        victims = np.empty(self.cap, np.int32)
        mo = ManageOut()
        pages = np.ascontiguousarray(self.host_pages) if self.P else np.zeros((1, 2, PART, D), np.uint16)
        self.lib.oracle_manage(self.h, _p(sel), k, t, _p(pages), _p(sel_slot), _p(sel_hit), _p(victims),
                               ctypes.byref(mo))
        return sel_slot[:k].copy(), sel_hit[:k].astype(bool), victims[:mo.evicted].copy(), mo

    def attend(self, sel: np.ndarray, sel_slot: np.ndarray, q_bits: np.ndarray) -> np.ndarray:
        sel = np.ascontiguousarray(sel, np.int32)
        sel_slot = np.ascontiguousarray(sel_slot, np.int32)
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        G = q_bits.shape[0]
        out = np.empty((G, D), np.float64)
        self.lib.oracle_attend_tail(self.h, _p(sel), _p(sel_slot), sel.shape[0], _p(q_bits), G,
                                    _p(self.tail), self.tail_n, _p(out))
        return out

    def clone_empty(self, cap: int) -> "TailUnit":
        """A unit with the same partitions, summaries, host pages and tail, and nothing resident."""
        c = TailUnit.__new__(TailUnit)
        c.lib, c.cap, c.ntok, c.P_cap = self.lib, cap, self.ntok, self.P_cap
        c.h = self.lib.oracle_unit_create_tail(self.P, max(self.P_cap, 1), cap)
        c.summ, c.host_pages = self.summ, self.host_pages
        c.tail, c.tail_n = self.tail.copy(), self.tail_n
        return c

    def step(self, q_bits: np.ndarray, k: int, t: int) -> dict:
        """Select over the complete partitions -> Manage/Retrieve -> Attention (with the tail)."""
        sc = scores(self.summ, q_bits, self.lib) if self.P else np.zeros(0)
        sel = topk(sc, k, self.lib) if self.P else np.zeros(0, np.int32)
        ss, hit, vic, mo = self.manage(sel, t)
        out = self.attend(sel, ss, q_bits)
        return dict(scores=sc, sel=sel, sel_slot=ss, sel_hit=hit, victims=vic, mo=mo, out=out)
