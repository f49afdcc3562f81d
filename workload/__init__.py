"""Seeded synthetic workloads for the SPIN sparse-decode data path.

The five workload shapes come from the decode configurations this library is
measured on: a tiny single-request case, a Qwen3-14B-shaped batch, a
Llama-3.1-70B-shaped batch, an eviction/metadata stress batch with variable
context, and a single 1M-token request. Only head shapes are taken from those
models; every value is drawn by ``gen.c`` (see its header for the recipe).

This package draws inputs only. It holds none of the method's arithmetic and is
shared by the oracle tests and by the CUDA path's tests and benchmark.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import sys
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libworkload.so")
_lock = threading.Lock()
_lib = None

D = 128
PART = 64


def build(force: bool = False) -> str:
    """Compile gen.c into libworkload.so next to it (gcc, OpenMP when available)."""
    src = os.path.join(_HERE, "gen.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", src, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("B", ctypes.c_int32),
        ("L", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("drift_a", ctypes.c_float),
        ("drift_c", ctypes.c_float),
        ("mu_std", ctypes.c_float),
        ("hot_norm", ctypes.c_float),
        ("hot_frac", ctypes.c_double),
        ("ctx_len", ctypes.POINTER(ctypes.c_int64)),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER
            L.wl_init.restype = None
            L.wl_ctx_partitions.restype = ctypes.c_int64
            L.wl_ctx_partitions.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            L.wl_query_init.argtypes = [P(_Cfg), ctypes.c_void_p]
            L.wl_query_step.argtypes = [P(_Cfg), ctypes.c_int32, ctypes.c_void_p]
            L.wl_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            L.wl_unit_mu.argtypes = [P(_Cfg), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_void_p]
            L.wl_unit_kv.argtypes = [P(_Cfg), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.wl_request_kv.argtypes = [P(_Cfg), ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int32]
            L.wl_unit_hot_count.restype = ctypes.c_int64
            L.wl_unit_hot_count.argtypes = [P(_Cfg), ctypes.c_int32]
            L.wl_unit_hot_mask.argtypes = [P(_Cfg), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            L.wl_normals.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
            L.wl_init()
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


@dataclasses.dataclass
class Workload:
    """One decode workload: shapes, policy knobs and the input recipe."""

    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    ctx_len: List[int]          # tokens per request
    topk: int                   # partitions selected per KV head
    buf_mult: int               # resident capacity = buf_mult * topk pages per KV head
    drift_a: float
    drift_c: float
    steps: int
    seed: int = 0
    mu_std: float = 0.5
    hot_norm: float = 0.0
    hot_frac: float = 0.0
    d: int = D
    part: int = PART
    mean_part: int = 0          # > 0: variable partitions averaging about this many tokens
    max_context: int = 0        # logical context capacity the deployment admits (0 = the longest context)

    # ---- derived shapes ----
    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def cap(self) -> int:
        return self.buf_mult * self.topk

    def partitions(self, b: int) -> int:
        return (self.ctx_len[b] + self.part - 1) // self.part

    @property
    def p_max(self) -> int:
        return max(self.partitions(b) for b in range(self.B))

    @property
    def units(self) -> int:
        return self.B * self.L * self.Hkv

    def host_kv_bytes(self) -> int:
        return sum(self.partitions(b) for b in range(self.B)) * self.L * self.Hkv * 2 * self.part * self.d * 2

    def selected_kv_bytes_per_step(self) -> int:
        return sum(min(self.topk, self.partitions(b)) for b in range(self.B)) * self.L * self.Hkv * 2 * self.part * self.d * 2

    def summary_bytes_per_step(self) -> int:
        return sum(self.partitions(b) for b in range(self.B)) * self.L * self.Hkv * self.d * 4

    # ---- variable partitions (a stand-in for a clustering Index) ----
    def var_partitions(self, b: int) -> int:
        """Partitions per KV head of request b when mean_part > 0 (the same for every head
        and layer of the request): ceil(ctx / mean_part), kept within [ceil(ctx / 64), ctx]."""
        n = self.ctx_len[b]
        if n == 0:
            return 0
        want = -(-n // max(self.mean_part, 1))
        return int(min(n, max(-(-n // self.part), want)))

    @property
    def max_partitions(self) -> int:
        return max((self.var_partitions(b) for b in range(self.B)), default=0)

    def unit_parts(self, layer: int, b: int, h: int):
        """Grouping of one unit's tokens: (order int32 [ctx], starts int32 [P + 1]).
        Partition p holds tokens order[starts[p]:starts[p + 1]]."""
        rng = np.random.default_rng([self.seed, 0x7061, layer, b, h])
        return random_parts(rng, self.ctx_len[b], self.var_partitions(b))

    def request_parts(self, layer: int, b: int):
        """unit_parts of every KV head of request b: order [Hkv][ctx], starts [Hkv][P + 1]."""
        parts = [self.unit_parts(layer, b, h) for h in range(self.Hkv)]
        return (np.stack([o for o, _ in parts]).astype(np.int32), np.stack([s for _, s in parts]).astype(np.int32))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ---- generator access ----
    def _cfg(self) -> _Cfg:
        self._ctx_arr = (ctypes.c_int64 * self.B)(*self.ctx_len)
        return _Cfg(self.seed, self.B, self.L, self.Hq, self.Hkv, self.d, self.drift_a, self.drift_c,
                    self.mu_std, self.hot_norm, self.hot_frac, self._ctx_arr)

    def request_kv(self, layer: int, b: int, k_out: Optional[np.ndarray] = None,
                   v_out: Optional[np.ndarray] = None, threads: int = 0):
        """bf16 bits [Hkv][ctx][128] of request b in `layer` (uint16 arrays)."""
        n = self.ctx_len[b]
        shape = (self.Hkv, n, self.d)
        k = k_out if k_out is not None else np.empty(shape, np.uint16)
        v = v_out if v_out is not None else np.empty(shape, np.uint16)
        assert k.shape == shape and v.shape == shape and k.dtype == np.uint16 and v.dtype == np.uint16
        cfg = self._cfg()
        lib().wl_request_kv(ctypes.byref(cfg), layer, b, _ptr(k), _ptr(v), threads)
        return k, v

    def unit_kv(self, layer: int, b: int, h: int, tok0: int = 0, ntok: Optional[int] = None):
        """bf16 bits [ntok][128] of K and V of one unit (layer, request, kv head)."""
        if ntok is None:
            ntok = self.ctx_len[b] - tok0
        k = np.empty((ntok, self.d), np.uint16)
        v = np.empty((ntok, self.d), np.uint16)
        cfg = self._cfg()
        lib().wl_unit_kv(ctypes.byref(cfg), layer, b, h, tok0, ntok, _ptr(k), _ptr(v))
        return k, v

    def unit_mu(self, layer: int, b: int, h: int) -> np.ndarray:
        P = self.partitions(b)
        mu = np.empty((P, self.d), np.float32)
        cfg = self._cfg()
        lib().wl_unit_mu(ctypes.byref(cfg), layer, b, h, 0, P, _ptr(mu))
        return mu

    def unit_hot_mask(self, layer: int, b: int, h: int) -> np.ndarray:
        m = np.zeros(self.partitions(b), np.uint8)
        cfg = self._cfg()
        lib().wl_unit_hot_mask(ctypes.byref(cfg), layer, b, h, _ptr(m))
        return m

    def queries(self) -> "QueryStream":
        return QueryStream(self)


class QueryStream:
    """Query trajectory q_t for all (layer, request, query head): fp32 state, bf16 output."""

    def __init__(self, w: Workload):
        self.w = w
        self.t = 0
        self.state = np.empty((w.L, w.B, w.Hq, w.d), np.float32)
        self._cfg = w._cfg()
        lib().wl_query_init(ctypes.byref(self._cfg), _ptr(self.state))

    def advance(self):
        self.t += 1
        lib().wl_query_step(ctypes.byref(self._cfg), self.t, _ptr(self.state))

    def bf16(self) -> np.ndarray:
        """Current step's queries as bf16 bits [L][B][Hq][128]."""
        out = np.empty(self.state.shape, np.uint16)
        lib().wl_to_bf16(_ptr(self.state), self.state.size, _ptr(out))
        return out


def random_parts(rng, n: int, P: int, window: int = 256, max_size: int = PART):
    """n tokens in P groups of 1..max_size: the tokens are shuffled within windows of
    `window` consecutive tokens (clusters gather nearby tokens, not only adjacent ones) and
    the order is cut into sizes drawn with exponential weights, so small and full groups
    both occur."""
    if n == 0:
        return np.zeros(0, np.int32), np.zeros(1, np.int32)
    assert 0 < P <= n <= max_size * P, (n, P)
    sizes = np.ones(P, np.int64)
    left = n - P
    w = rng.exponential(size=P)
    add = np.minimum(max_size - 1, np.floor(left * w / w.sum()).astype(np.int64))
    sizes += add
    left -= int(add.sum())
    while left > 0:  # the remainder, one token each to groups with room, in random order
        room = rng.permutation(np.flatnonzero(sizes < max_size))[:left]
        sizes[room] += 1
        left -= len(room)
    order = np.concatenate([t0 + rng.permutation(min(window, n - t0)) for t0 in range(0, n, window)])
    starts = np.concatenate([[0], np.cumsum(sizes)])
    return order.astype(np.int32), starts.astype(np.int32)


def normals(seed: int, tag: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().wl_normals(seed, tag, n, _ptr(out))
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# The decode workloads.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """1 request, 1 layer, 4 query / 4 KV heads, 4096 tokens, top-8 of 64, 40 pages/head, 16 steps."""
    return Workload("tiny", B=1, L=1, Hq=4, Hkv=4, ctx_len=[4096], topk=8, buf_mult=5,
                    drift_a=0.9, drift_c=0.1, steps=16, seed=seed)


def qwen3_14b(seed: int = 0) -> Workload:
    """Qwen3-14B-shaped decode: 40 q / 8 kv heads, 8 layers, batch 32, 32K context, top-32, 5x buffer, 64 steps;
    logical capacity 131072 tokens (the model's extended context)."""
    return Workload("qwen3_14b_32k", B=32, L=8, Hq=40, Hkv=8, ctx_len=[32768] * 32, topk=32, buf_mult=5,
                    drift_a=0.9, drift_c=0.1, steps=64, seed=seed, max_context=131072)


def llama31_70b(seed: int = 0) -> Workload:
    """Llama-3.1-70B-shaped decode: 64 q / 8 kv heads, 4 layers, batch 16, 128K context, top-64, 5x, 32 steps;
    logical capacity 131072 tokens (the model's context)."""
    return Workload("llama31_70b_128k", B=16, L=4, Hq=64, Hkv=8, ctx_len=[131072] * 16, topk=64, buf_mult=5,
                    drift_a=0.8, drift_c=0.2, steps=32, seed=seed, max_context=131072)


def stress(buf_mult: int = 1, seed: int = 0) -> Workload:
    """Qwen3-32B-shaped eviction/metadata stress: 64 q / 8 kv heads, 1 layer, batch 256,
    context uniform over whole partitions in [8192, 32768] tokens, top-16, 1x or 5x buffer, 32 steps;
    logical capacity 131072 tokens (the model's extended context)."""
    ctx = [64 * int(lib().wl_ctx_partitions(seed, b, 128, 512)) for b in range(256)]
    return Workload(f"stress_m{buf_mult}", B=256, L=1, Hq=64, Hkv=8, ctx_len=ctx, topk=16, buf_mult=buf_mult,
                    drift_a=0.7, drift_c=0.3, steps=32, seed=seed, max_context=131072)


def long_1m(seed: int = 0) -> Workload:
    """Single 1M-token request: 40 q / 8 kv heads, 1 layer, 16384 partitions/head, top-128, 5x,
    1% of partitions offset by 3 * (normalised group query at step 0), drift 0.95/0.05, 64 steps."""
    return Workload("long_1m", B=1, L=1, Hq=40, Hkv=8, ctx_len=[1048576], topk=128, buf_mult=5,
                    drift_a=0.95, drift_c=0.05, steps=64, seed=seed, hot_norm=3.0, hot_frac=0.01, max_context=1048576)


ALL = {"tiny": tiny, "qwen3_14b_32k": qwen3_14b, "llama31_70b_128k": llama31_70b,
       "stress_m1": lambda seed=0: stress(1, seed), "stress_m5": lambda seed=0: stress(5, seed),
       "long_1m": long_1m}


def by_name(name: str, seed: int = 0) -> Workload:
    return ALL[name](seed)
