"""A Python handle around one spin_ctx (marshalling only; every step runs in libspin.so).

PyTorch supplies device memory and streams; numpy supplies host buffers.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import _binding as B


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class SpinContext:
    """Owns one library context: configuration, offload, decode steps, stats, state export."""

    def __init__(self, batch: int, layers: int, q_heads: int, kv_heads: int, ctx_len: Sequence[int], topk: int,
                 buf_mult: int, device: int = 0, seg_pool_segments: int = 0, flags: int = 0,
                 append_tokens: int = 0, max_partitions: int = 0, max_context: int = 0):
        self.B, self.L, self.Hq, self.Hkv = batch, layers, q_heads, kv_heads
        self.G = q_heads // kv_heads
        self.ctx_len = [int(x) for x in ctx_len]
        self.k, self.buf_mult = topk, buf_mult
        self.cap = topk * buf_mult
        self.append_tokens = int(append_tokens)
        self.tail_mode = self.append_tokens > 0
        self.max_partitions = int(max_partitions)
        self.part_mode = self.max_partitions > 0
        PT = B.PART_TOKENS
        if self.part_mode:
            # variable partitions: none until each (layer, request) is offloaded
            self.P = [0] * batch
            self.P_cap = [self.max_partitions] * batch
        elif self.tail_mode:
            # complete partitions per (layer, request); the rest of the context is the tail
            self.P = [n // PT for n in self.ctx_len]
            self.P_cap = [(n + self.append_tokens + PT - 1) // PT for n in self.ctx_len]
        else:
            self.P = [(n + PT - 1) // PT for n in self.ctx_len]
            self.P_cap = list(self.P)
        self.P_lb = [list(self.P) for _ in range(layers)]
        self.tail_lb = [[(n % PT) if self.tail_mode else 0 for n in self.ctx_len] for _ in range(layers)]
        self.P_max = max(self.P_cap) if self.P_cap else 0
        if self.part_mode:
            self.P_lb = [[0] * batch for _ in range(layers)]
        self.device = device
        self._ctx_arr = (ctypes.c_int64 * batch)(*self.ctx_len)
        cfg = B.spin_config(batch, layers, q_heads, kv_heads, B.HEAD_DIM, B.PART_TOKENS, topk, buf_mult,
                            self._ctx_arr, 0, seg_pool_segments, device, flags, self.append_tokens,
                            self.max_partitions, int(max_context))
        self.h = B.spin_create(cfg)

    @classmethod
    def for_workload(cls, w, device: int = 0, **kw) -> "SpinContext":
        """A context for a workload; variable partitions when the workload has mean_part > 0."""
        if getattr(w, "mean_part", 0) and "max_partitions" not in kw:
            kw["max_partitions"] = w.max_partitions
        if getattr(w, "max_context", 0) and "max_context" not in kw:
            kw["max_context"] = w.max_context
        return cls(w.B, w.L, w.Hq, w.Hkv, w.ctx_len, w.topk, w.buf_mult, device=device, **kw)

    def close(self):
        if getattr(self, "h", None):
            B.spin_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---- Index + Offload ----
    def index_offload_host(self, b: int, layer: int, k_bits: np.ndarray, v_bits: np.ndarray, stream: int = 0):
        """k_bits, v_bits: uint16 [Hkv][ctx_len[b]][128] host arrays (kept alive until the stream syncs)."""
        n = self.ctx_len[b]
        assert k_bits.shape == (self.Hkv, n, B.HEAD_DIM) and v_bits.shape == k_bits.shape
        B.spin_index_offload(self.h, b, layer, _ptr(k_bits), _ptr(v_bits), n, True, stream)

    def index_offload_device(self, b: int, layer: int, k_dev, v_dev, stream: int = 0):
        """k_dev, v_dev: contiguous CUDA tensors [Hkv][ctx_len[b]][128] of bf16 or int16 bits."""
        n = self.ctx_len[b]
        B.spin_index_offload(self.h, b, layer, k_dev.data_ptr(), v_dev.data_ptr(), n, False, stream)

    def index_offload_parts(self, b: int, layer: int, k, v, order: np.ndarray, starts: np.ndarray,
                            stream: int = 0):
        """Variable partitions. k, v: uint16 host arrays or CUDA tensors [Hkv][ctx_len[b]][128];
        order int32 [Hkv][ctx_len[b]] and starts int32 [Hkv][P + 1] host arrays (the grouping:
        partition p of head h holds tokens order[h][starts[h][p]:starts[h][p + 1]]).
        Returns once done."""
        n = self.ctx_len[b]
        order = np.ascontiguousarray(order, np.int32)
        starts = np.ascontiguousarray(starts, np.int32)
        assert order.shape == (self.Hkv, n) and starts.ndim == 2 and starts.shape[0] == self.Hkv
        n_parts = starts.shape[1] - 1
        host = isinstance(k, np.ndarray)
        kp = _ptr(k) if host else k.data_ptr()
        vp = _ptr(v) if host else v.data_ptr()
        if host:
            assert k.shape == (self.Hkv, n, B.HEAD_DIM) and v.shape == k.shape
        B.spin_index_offload_parts(self.h, b, layer, kp, vp, n, _ptr(order), _ptr(starts), n_parts, host, stream)
        self.P_lb[layer][b] = n_parts

    # ---- KV append (tail mode) ----
    def append_kv(self, layer: int, k_dev, v_dev, stream: int = 0):
        """One new token per request: k_dev, v_dev CUDA bf16/int16 [B][Hkv][128]."""
        B.spin_append_kv(self.h, layer, k_dev.data_ptr(), v_dev.data_ptr(), stream)
        for b in range(self.B):
            self.tail_lb[layer][b] += 1
            if self.tail_lb[layer][b] == B.PART_TOKENS:
                self.tail_lb[layer][b] = 0
                self.P_lb[layer][b] += 1

    # ---- buffer elasticity ----
    def set_buffer(self, b: int, pages: int, stream: int = 0):
        """Resident budget of request b: topk <= pages <= buf_mult * topk pages per unit."""
        B.spin_set_buffer(self.h, b, pages, stream)

    # ---- decode ----
    def decode_step(self, layer: int, q_dev, out_dev, stream: int = 0):
        """q_dev: CUDA bf16/int16 [B][Hq][128]; out_dev: CUDA fp32 [B][Hq][128]."""
        B.spin_decode_step(self.h, layer, q_dev.data_ptr(), out_dev.data_ptr(), stream)

    def decode_step_host(self, layer: int, q_host_ptr: int, out_host_ptr: int, stream: int = 0):
        B.spin_decode_step_host(self.h, layer, q_host_ptr, out_host_ptr, stream)

    # ---- inspection ----
    def stats(self, check: bool = True) -> dict:
        st = B.spin_stats(self.h, check=check)
        d = st.as_dict()
        d["rc"] = st.rc
        return d

    def export(self, layer: int, resolve: bool = True, scores: bool = False) -> dict:
        Ul = self.B * self.Hkv
        out = dict(
            keff=np.empty(Ul, np.int32),
            sel=np.empty((Ul, self.k), np.int32),
            sel_slot=np.empty((Ul, self.k), np.int32),
            sel_hit=np.empty((Ul, self.k), np.uint8),
            slot_part=np.empty((Ul, self.cap), np.int32),
            last_use=np.empty((Ul, self.cap), np.int32),
            unit_info=np.empty((Ul, 8), np.int32),
        )
        if resolve:
            out["resolve"] = np.empty((Ul, max(self.P_max, 1)), np.int32)
            out["live_segs"] = np.empty(Ul, np.int32)
        if scores:
            out["scores"] = np.empty((Ul, max(self.P_max, 1)), np.float32)
        v = B.spin_state_view(*[(_ptr(out[n]) if n in out else None) for n, _ in B.spin_state_view._fields_])
        B.spin_debug_export(self.h, layer, v)
        return out

    def read_tail(self, layer: int, b: int, h: int) -> np.ndarray:
        """The unit's tail page (tail mode): [2][64][128] bf16 bits."""
        return self.read_page(layer, b, h, self.cap)

    def read_page(self, layer: int, b: int, h: int, slot: int) -> np.ndarray:
        dst = np.empty((2, B.PART_TOKENS, B.HEAD_DIM), np.uint16)
        B.spin_debug_read_page(self.h, layer, b, h, slot, _ptr(dst))
        return dst

    def summaries(self, layer: int, b: int, h: int) -> np.ndarray:
        P = self.P_lb[layer][b]
        dst = np.empty((max(P, 1), B.HEAD_DIM), np.float32)
        B.spin_debug_summaries(self.h, layer, b, h, _ptr(dst))
        return dst[:P]
