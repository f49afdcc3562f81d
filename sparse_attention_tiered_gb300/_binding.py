"""ctypes binding of libspin.so (argument marshalling only).

Every function here has the name of the C entry point it wraps (include/spin.h)
and does nothing but convert arguments. All computation happens in the CUDA
library; when libspin.so is missing or cannot be loaded, these calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None

SPIN_OK = 0
SPIN_ERR_INVALID = 1
SPIN_ERR_CUDA = 2
SPIN_ERR_OOM = 3
SPIN_ERR_CAPACITY = 4
SPIN_ERR_TIMEOUT = 5
SPIN_ERR_STATE = 6
STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "CUDA", 3: "OOM", 4: "CAPACITY", 5: "TIMEOUT", 6: "STATE"}

SPIN_FLAG_STAGE_TIMING = 1 << 0
SPIN_FLAG_TIER_SPLIT = 1 << 2
SPIN_FLAG_HOST_HUGEPAGES = 1 << 3
SPIN_FLAG_PHASED = 1 << 4
SPIN_FLAG_TEST_FAIL_PINNED = 1 << 16
SPIN_FLAG_TEST_NO_RETRIEVE = 1 << 17

HEAD_DIM = 128
PART_TOKENS = 64
PAGE_BYTES = 32768
SPIN_NOALLOC_MAX_SCORES_DEFAULT = 1 << 20  # SPIN_NOALLOC_MAX_SCORES in include/spin.h

# Every symbol include/spin.h declares.
EXPORTS = ("spin_create", "spin_index_offload", "spin_index_offload_parts", "spin_append_kv", "spin_set_buffer", "spin_decode_step", "spin_decode_step_host", "spin_stats",
           "spin_debug_export", "spin_debug_read_page", "spin_debug_summaries", "spin_destroy", "spin_last_error",
           "spin_select_noalloc", "spin_measure_host_read")


class SpinError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"SPIN_ERR_{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class spin_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("layers", ctypes.c_int32),
        ("q_heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("part_tokens", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("buf_mult", ctypes.c_int32),
        ("ctx_len", ctypes.POINTER(ctypes.c_int64)),
        ("seg_entries", ctypes.c_int32),
        ("seg_pool_segments", ctypes.c_int64),
        ("device", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("append_tokens", ctypes.c_int32),
        ("max_partitions", ctypes.c_int32),
        ("max_context", ctypes.c_int64),
    ]


class spin_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "steps", "hits", "misses", "evictions", "lru_rounds", "retrieved_bytes", "selected_bytes",
        "live_segments", "pool_segments", "metadata_bytes", "flat_table_bytes", "hbm_pool_bytes",
        "host_store_bytes", "summary_bytes", "timed_calls")] + [
        (n, ctypes.c_double) for n in ("ms_score", "ms_manage", "ms_pages", "ms_combine", "ms_kernel")] + [
        ("device_error", ctypes.c_uint32), ("appended_tokens", ctypes.c_int64), ("tail_flushes", ctypes.c_int64)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class spin_state_view(ctypes.Structure):
    _fields_ = [
        ("keff", ctypes.c_void_p),
        ("sel", ctypes.c_void_p),
        ("sel_slot", ctypes.c_void_p),
        ("sel_hit", ctypes.c_void_p),
        ("slot_part", ctypes.c_void_p),
        ("last_use", ctypes.c_void_p),
        ("resolve", ctypes.c_void_p),
        ("live_segs", ctypes.c_void_p),
        ("unit_info", ctypes.c_void_p),
        ("scores", ctypes.c_void_p),
    ]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libspin.so (building it first when it is missing or stale and nvcc is present)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libspin.so not found at {path}; run __graft_entry__.build()")
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.spin_create.argtypes = [ctypes.POINTER(spin_config), ctypes.POINTER(vp)]
            L.spin_create.restype = ctypes.c_int
            L.spin_index_offload.argtypes = [vp, i32, i32, vp, vp, i64, i32, vp]
            L.spin_index_offload.restype = ctypes.c_int
            L.spin_index_offload_parts.argtypes = [vp, i32, i32, vp, vp, i64, vp, vp, i32, i32, vp]
            L.spin_index_offload_parts.restype = ctypes.c_int
            L.spin_append_kv.argtypes = [vp, i32, vp, vp, vp]
            L.spin_append_kv.restype = ctypes.c_int
            L.spin_set_buffer.argtypes = [vp, i32, i32, vp]
            L.spin_set_buffer.restype = ctypes.c_int
            L.spin_decode_step.argtypes = [vp, i32, vp, vp, vp]
            L.spin_decode_step.restype = ctypes.c_int
            L.spin_decode_step_host.argtypes = [vp, i32, vp, vp, vp]
            L.spin_decode_step_host.restype = ctypes.c_int
            L.spin_stats.argtypes = [vp, ctypes.POINTER(spin_stats_t)]
            L.spin_stats.restype = ctypes.c_int
            L.spin_debug_export.argtypes = [vp, i32, ctypes.POINTER(spin_state_view)]
            L.spin_debug_export.restype = ctypes.c_int
            L.spin_debug_read_page.argtypes = [vp, i32, i32, i32, i32, vp]
            L.spin_debug_read_page.restype = ctypes.c_int
            L.spin_debug_summaries.argtypes = [vp, i32, i32, i32, vp]
            L.spin_debug_summaries.restype = ctypes.c_int
            L.spin_destroy.argtypes = [vp]
            L.spin_destroy.restype = None
            L.spin_select_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
            L.spin_select_noalloc.restype = ctypes.c_int
            L.spin_measure_host_read.argtypes = [vp, i64, i32, ctypes.POINTER(ctypes.c_double), vp]
            L.spin_measure_host_read.restype = ctypes.c_int
            L.spin_last_error.argtypes = [vp]
            L.spin_last_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(rc: int, ctx=None):
    if rc != SPIN_OK:
        msg = load().spin_last_error(ctx)
        raise SpinError(rc, msg.decode(errors="replace") if msg else "")


# ---------------------------------------------------------------------------
# Thin wrappers with the C names. Pointers are ints (device or host addresses).
# ---------------------------------------------------------------------------

def spin_create(cfg: spin_config) -> int:
    h = ctypes.c_void_p()
    _check(load().spin_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def spin_index_offload(ctx: int, b: int, layer: int, k_ptr: int, v_ptr: int, n_tokens: int, src_is_host: bool,
                       stream: int = 0):
    _check(load().spin_index_offload(ctx, b, layer, k_ptr, v_ptr, n_tokens, 1 if src_is_host else 0, stream), ctx)


def spin_index_offload_parts(ctx: int, b: int, layer: int, k_ptr: int, v_ptr: int, n_tokens: int, order_ptr: int,
                             starts_ptr: int, n_parts: int, src_is_host: bool, stream: int = 0):
    _check(load().spin_index_offload_parts(ctx, b, layer, k_ptr, v_ptr, n_tokens, order_ptr, starts_ptr, n_parts,
                                           1 if src_is_host else 0, stream), ctx)


def spin_append_kv(ctx: int, layer: int, k_ptr: int, v_ptr: int, stream: int = 0):
    _check(load().spin_append_kv(ctx, layer, k_ptr, v_ptr, stream), ctx)


def spin_set_buffer(ctx: int, b: int, pages: int, stream: int = 0):
    _check(load().spin_set_buffer(ctx, b, pages, stream), ctx)


def spin_decode_step(ctx: int, layer: int, q_ptr: int, out_ptr: int, stream: int = 0):
    _check(load().spin_decode_step(ctx, layer, q_ptr, out_ptr, stream), ctx)


def spin_decode_step_host(ctx: int, layer: int, q_host_ptr: int, out_host_ptr: int, stream: int = 0):
    _check(load().spin_decode_step_host(ctx, layer, q_host_ptr, out_host_ptr, stream), ctx)


def spin_stats(ctx: int, check: bool = True) -> spin_stats_t:
    st = spin_stats_t()
    rc = load().spin_stats(ctx, ctypes.byref(st))
    if check:
        _check(rc, ctx)
    st.rc = rc
    return st


def spin_debug_export(ctx: int, layer: int, view: spin_state_view):
    _check(load().spin_debug_export(ctx, layer, ctypes.byref(view)), ctx)


def spin_debug_read_page(ctx: int, layer: int, b: int, h: int, slot: int, dst_ptr: int):
    _check(load().spin_debug_read_page(ctx, layer, b, h, slot, dst_ptr), ctx)


def spin_debug_summaries(ctx: int, layer: int, b: int, h: int, dst_ptr: int):
    _check(load().spin_debug_summaries(ctx, layer, b, h, dst_ptr), ctx)


def spin_select_noalloc(summ_ptr: int, q_ptr: int, units: int, parts: int, group: int, topk: int, sel_ptr: int,
                        stream: int = 0):
    _check(load().spin_select_noalloc(summ_ptr, q_ptr, units, parts, group, topk, sel_ptr, stream))


def spin_destroy(ctx: int):
    load().spin_destroy(ctx)


def spin_measure_host_read(host_ptr: int, nbytes: int, ctas_per_sm: int = 1, stream: int = 0) -> float:
    """GB/s of SM zero-copy reads of a pinned host buffer (see include/spin.h)."""
    g = ctypes.c_double(0.0)
    _check(load().spin_measure_host_read(host_ptr, nbytes, ctas_per_sm, ctypes.byref(g), stream))
    return g.value


def spin_last_error(ctx=None) -> str:
    m = load().spin_last_error(ctx)
    return m.decode(errors="replace") if m else ""
