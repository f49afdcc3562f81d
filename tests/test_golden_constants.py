"""The design constants the pages state (tests/golden/page_constants.txt) against the
oracle's, the library's and the workloads' own values."""
import os
import re

import oracle as O
import workload as W

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    out = {}
    with open(os.path.join(HERE, "golden", "page_constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, value, cite = line.split(None, 2)
                assert cite.startswith("[XT]") or cite.startswith("[GS]"), f"{name} has no citation"
                out[name] = int(value)
    return out


def oracle_defines():
    with open(os.path.join(os.path.dirname(O.__file__), "spin_oracle.c")) as f:
        return {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define (\w+) (\d+)", f.read(), re.M)}


def test_oracle_uses_the_pages_bucket_count():
    assert oracle_defines()["OBUCKETS"] == golden()["lru_buckets"]


def test_workloads_use_the_pages_buffer_multiple():
    g = golden()["buffer_multiple"]
    for make in (W.tiny, W.qwen3_14b, W.llama31_70b, W.long_1m):
        assert make().buf_mult == g, make.__name__
    assert W.stress(buf_mult=5).buf_mult == g


def test_library_uses_the_pages_bucket_count():
    with open(os.path.join(os.path.dirname(HERE), "include", "spin.h")) as f:
        m = re.search(r"^#define SPIN_LRU_BUCKETS (\d+)", f.read(), re.M)
    assert m and int(m.group(1)) == golden()["lru_buckets"]


def test_boundary_covers_the_pages_operations():
    """The five operations each have an entry point or a kernel stage behind the C ABI:
    Index + Offload (spin_index_offload, spin_index_offload_parts), Select, Retrieve and
    Attention (the stages of spin_decode_step)."""
    with open(os.path.join(os.path.dirname(HERE), "include", "spin.h")) as f:
        h = f.read()
    assert golden()["pipeline_operations"] == 5
    for name in ("spin_index_offload", "spin_index_offload_parts", "spin_decode_step"):
        assert re.search(r"^int " + name + r"\(", h, re.M), name
    for op in ("Index", "Offload", "Select", "Retrieve", "Attention"):
        assert op in h, op
