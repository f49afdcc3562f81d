"""The C ABI library without a GPU: it loads, exports every declared symbol and
fails cleanly (status codes, messages) where a device would be needed."""
import ctypes
import os
import re

import pytest

import sparse_attention_tiered_gb300 as spin
from sparse_attention_tiered_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^(?:int|void|const char\*)\s+(spin_\w+)\s*\(", txt, re.M)
    return sorted(set(names))


def test_header_declares_the_bound_entry_points():
    assert sorted(B.EXPORTS) == declared_symbols()


def test_library_loads_and_exports_every_symbol():
    lib = spin.load()
    for name in declared_symbols():
        assert hasattr(lib, name), f"libspin.so does not export {name}"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def _cfg(**kw):
    ctx = (ctypes.c_int64 * 2)(4096, 4096)
    d = dict(batch=2, layers=1, q_heads=8, kv_heads=2, head_dim=128, part_tokens=64, topk=8, buf_mult=5,
             ctx_len=ctx, seg_entries=0, seg_pool_segments=0, device=0, flags=0)
    d.update(kw)
    c = B.spin_config(**{k: v for k, v in d.items()})
    c._keep = ctx
    return c


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(part_tokens=32), dict(q_heads=7), dict(topk=0),
                                 dict(topk=1000), dict(buf_mult=0), dict(batch=0), dict(seg_entries=16),
                                 dict(q_heads=2 * 17, kv_heads=2), dict(seg_pool_segments=-1),
                                 dict(append_tokens=-1), dict(append_tokens=1 << 30), dict(max_partitions=-1),
                                 dict(max_partitions=(1 << 20) + 1), dict(max_partitions=100, append_tokens=10),
                                 dict(max_partitions=63)])
def test_invalid_configs_are_rejected(bad):
    with pytest.raises(B.SpinError) as e:
        B.spin_create(_cfg(**bad))
    assert e.value.code == B.SPIN_ERR_INVALID
    assert B.spin_last_error(None)


def test_negative_context_rejected():
    ctx = (ctypes.c_int64 * 2)(-1, 64)
    with pytest.raises(B.SpinError) as e:
        B.spin_create(_cfg(ctx_len=ctx))
    assert e.value.code == B.SPIN_ERR_INVALID


def test_injected_pinned_failure_reports_oom():
    with pytest.raises(B.SpinError) as e:
        B.spin_create(_cfg(flags=B.SPIN_FLAG_TEST_FAIL_PINNED))
    assert e.value.code == B.SPIN_ERR_OOM
    assert "pinned" in B.spin_last_error(None)


def test_null_arguments():
    lib = spin.load()
    assert lib.spin_create(None, None) == B.SPIN_ERR_INVALID
    assert lib.spin_decode_step(None, 0, None, None, None) == B.SPIN_ERR_INVALID
    assert lib.spin_stats(None, None) == B.SPIN_ERR_INVALID
    assert lib.spin_index_offload_parts(None, 0, 0, None, None, 0, None, None, 0, 0, None) == B.SPIN_ERR_INVALID
    lib.spin_destroy(None)


def test_create_without_gpu_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(B.SpinError) as e:
        B.spin_create(_cfg())
    assert e.value.code in (B.SPIN_ERR_CUDA, B.SPIN_ERR_OOM)
