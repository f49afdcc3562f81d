"""The N > 1 benchmark path on CPU: two gloo ranks.

Ranks run independent batches (rank r draws its workload with seed r); the only
collectives are a barrier and the max over ranks of the timed region.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    import workload as W
    R = bench.Ranks()
    R.init("gloo")
    R.barrier()
    ms = 10.0 + 5.0 * rank                       # the slower rank sets the job time
    m = R.max(ms)
    args = type("A", (), {"workload": "tiny", "layers": 0, "batch": 0})()
    w = bench.make_workload(args, R.rank)
    k, _ = w.unit_kv(0, 0, 0, 0, 64)
    q.put((rank, m, bench.job_tokens_per_s(w.B * 10, R.world, m), w.seed, k.tobytes()))
    R.barrier()
    R.close()


def test_two_gloo_ranks_max_timing_and_disjoint_shards():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, v0, s0, k0), (r1, m1, v1, s1, k1) = res
    assert m0 == m1 == 15.0                      # max over ranks
    assert v0 == v1 == pytest.approx(1 * 10 * 2 / 15e-3)
    assert (s0, s1) == (0, 1) and k0 != k1       # independent shards


def test_single_rank_defaults():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    R = bench.Ranks()
    assert (R.world, R.rank) == (1, 0)
    assert R.max(3.5) == 3.5
    assert bench.job_tokens_per_s(32, 1, 2.0) == pytest.approx(16000.0)


def _mem_worker(rank, world, port, avail, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    R = bench.Ranks()
    R.init("gloo")
    need = (10 + rank) << 30  # 10 and 11 GiB of page store
    try:
        tot, av = R.check_host_memory(need, avail_bytes=avail + rank * (1 << 30))
        q.put((rank, "ok", tot, av))
    except SystemExit as e:
        q.put((rank, "refused", str(e), None))
    R.barrier()
    R.close()


@pytest.mark.parametrize("avail_gib,expect", [(40, "ok"), (20, "refused")])
def test_two_gloo_ranks_host_memory_check(avail_gib, expect):
    """Both ranks' page stores (21 GiB together) against the node's available memory (the
    smaller rank report, 90% usable): the same decision on every rank, with the figures."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_mem_worker, args=(r, world, port, avail_gib << 30, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [expect, expect]
    if expect == "ok":
        assert res[0][2] == res[1][2] == float(21 << 30) and res[0][3] == float(avail_gib << 30)
    else:
        assert "21.0 GiB" in res[0][2] and "20.0 GiB available" in res[0][2]


def test_gpu_local_cpus_from_sysfs(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    d = tmp_path / "bus" / "pci" / "devices" / "0000:00:07.0"
    d.mkdir(parents=True)
    (d / "local_cpulist").write_text("0-3,8,10-11\n")
    assert bench.gpu_local_cpus("0000:00:07.0", sysfs=str(tmp_path)) == {0, 1, 2, 3, 8, 10, 11}
    assert bench.gpu_local_cpus("0000:00:08.0", sysfs=str(tmp_path)) is None
    assert bench.parse_cpulist("5") == {5}
    meminfo = tmp_path / "meminfo"
    meminfo.write_text("MemTotal: 100 kB\nMemAvailable:    2048 kB\n")
    assert bench.mem_available_bytes(str(meminfo)) == 2048 * 1024
