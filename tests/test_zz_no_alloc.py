"""spin_select_noalloc: the allocation-free Select entry point.

It serves callers that cannot allocate device memory (graph capture in progress,
an engine whose allocator owns the device, hosts that forbid run-time
allocation). Its output must equal the selection the regular decode step makes
for the same summaries and queries. Collected last (file name) so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import workload as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _layer_summaries(ctx, w, layer):
    return np.stack([ctx.summaries(layer, b, h) for b in range(w.B) for h in range(w.Hkv)])


def test_select_noalloc_matches_decode_step_selection():
    import sparse_attention_tiered_gb300 as spin
    from sparse_attention_tiered_gb300 import SpinContext

    w = W.Workload("noalloc", B=3, L=1, Hq=10, Hkv=2, ctx_len=[4096] * 3, topk=8, buf_mult=2,
                   drift_a=0.8, drift_c=0.2, steps=2, seed=31)
    lib = spin.load()
    U, P = w.B * w.Hkv, w.partitions(0)
    with SpinContext.for_workload(w) as ctx:
        for b in range(w.B):
            k, v = w.request_kv(0, b)
            ctx.index_offload_host(b, 0, k, v)
            torch.cuda.synchronize()
        summ = torch.from_numpy(_layer_summaries(ctx, w, 0)).cuda().contiguous()  # [U][P][128]
        qs = w.queries()
        out = torch.empty((w.B, w.Hq, 128), dtype=torch.float32, device="cuda")
        for call in range(2):  # two calls in a row, each against that step's decode selection
            q = torch.from_numpy(qs.bf16()[0].view(np.int16)).cuda()   # [B][Hq][128] == [U][G][128]
            ctx.decode_step(0, q, out)
            torch.cuda.synchronize()
            ref = ctx.export(0, resolve=False)["sel"]
            sel = torch.full((U, w.topk), -7, dtype=torch.int32, device="cuda")
            rc = lib.spin_select_noalloc(summ.data_ptr(), q.data_ptr(), U, P, w.G, w.topk, sel.data_ptr(), None)
            assert rc == 0, spin.spin_last_error(None)
            torch.cuda.synchronize()
            assert np.array_equal(sel.cpu().numpy(), ref), f"call {call}: selections differ"
            qs.advance()


def test_select_noalloc_short_units_pad_and_limits():
    import sparse_attention_tiered_gb300 as spin
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_INVALID, SPIN_NOALLOC_MAX_SCORES_DEFAULT

    lib = spin.load()
    U, P, G, k = 2, 3, 1, 5                 # fewer partitions than k: the tail is -1
    summ = torch.zeros((U, P, 128), dtype=torch.float32, device="cuda")
    summ[:, :, 0] = torch.tensor([[1.0, 3.0, 2.0], [5.0, 5.0, -1.0]], device="cuda")
    q = torch.zeros((U, G, 128), dtype=torch.int16, device="cuda")
    q[:, :, 0] = 0x3F80                     # bf16 1.0: the score is the first summary coordinate
    sel = torch.empty((U, k), dtype=torch.int32, device="cuda")
    assert lib.spin_select_noalloc(summ.data_ptr(), q.data_ptr(), U, P, G, k, sel.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert sel.cpu().tolist() == [[0, 1, 2, -1, -1], [0, 1, 2, -1, -1]]
    sel2 = torch.empty((U, 2), dtype=torch.int32, device="cuda")
    assert lib.spin_select_noalloc(summ.data_ptr(), q.data_ptr(), U, P, G, 2, sel2.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert sel2.cpu().tolist() == [[1, 2], [0, 1]]     # equal scores go to the lower index
    # sizes beyond the static scratch are refused, with a message
    big = SPIN_NOALLOC_MAX_SCORES_DEFAULT // 1024 + 1
    rc = lib.spin_select_noalloc(summ.data_ptr(), q.data_ptr(), big, 1024, G, k, sel.data_ptr(), None)
    assert rc == SPIN_ERR_INVALID and "scratch" in spin.spin_last_error(None)


def _noalloc(summ, q, topk):
    import sparse_attention_tiered_gb300 as spin
    lib = spin.load()
    U, P, G = summ.shape[0], summ.shape[1], q.shape[1]
    sd = torch.from_numpy(np.ascontiguousarray(summ, np.float32)).cuda()
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda()
    sel = torch.full((U, topk), -7, dtype=torch.int32, device="cuda")
    rc = lib.spin_select_noalloc(sd.data_ptr(), qd.data_ptr(), U, P, G, topk, sel.data_ptr(), None)
    assert rc == 0, spin.spin_last_error(None)
    torch.cuda.synchronize()
    return sel.cpu().numpy()


@pytest.mark.parametrize("P", [513, 5000, 32768])
def test_select_noalloc_ties_across_warp_ranges(P):
    """Exact scores (q = e_0, so the score is the summary's first coordinate) with copies of
    the k-th value planted across the boundaries of the per-warp key ranges: the selection
    equals a stable argsort of -score (equal scores to the lower index), first k, ascending.
    P = 513 and 32768 take the warp-scan compaction, P = 5000 the wide-unit paths."""
    rng = np.random.default_rng(P)
    U, G, k = 2, 1, 64
    vals = rng.standard_normal((U, P)).astype(np.float32)
    chunk = -(-P // 512) * 32  # keys per warp range of the 512-thread compaction
    for u in range(U):
        thr = vals[u, np.argsort(-vals[u], kind="stable")[k - 1]]
        for m in range(chunk, P, chunk):
            for dlt in (-2, -1, 0, 1):
                if 0 <= m + dlt < P:
                    vals[u, m + dlt] = thr
    summ = np.zeros((U, P, 128), np.float32)
    summ[:, :, 0] = vals
    q = np.zeros((U, G, 128), np.uint16)
    q[:, :, 0] = 0x3F80  # bf16 1.0
    got = _noalloc(summ, q, k)
    for u in range(U):
        ref = np.sort(np.argsort(-vals[u], kind="stable")[:k])
        assert np.array_equal(got[u], ref), (u, np.setdiff1d(got[u], ref), np.setdiff1d(ref, got[u]))


@pytest.mark.parametrize("P", [512, 16384])
def test_select_noalloc_matches_oracle(P):
    """Against the oracle's double-precision scores and top-k, with the 1e-5 relative tie band."""
    import oracle as O
    from parity import check_selection
    rng = np.random.default_rng(7 + P)
    U, G, k = 4, 5, 32
    summ = (0.5 * rng.standard_normal((U, P, 128))).astype(np.float32)
    qf = rng.standard_normal((U, G, 128)).astype(np.float32)
    q = ((qf.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)  # bf16 bits (round half up)
    got = _noalloc(summ, q, k)
    for u in range(U):
        sc = O.scores(summ[u].astype(np.float64), q[u])
        check_selection(sc, O.topk(sc, k), got[u], f"unit {u}")


def test_select_noalloc_refuses_too_many_partitions():
    import sparse_attention_tiered_gb300 as spin
    from sparse_attention_tiered_gb300._binding import SPIN_ERR_INVALID
    lib = spin.load()
    summ = torch.zeros((1, 16, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((1, 1, 128), dtype=torch.int16, device="cuda")
    sel = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    rc = lib.spin_select_noalloc(summ.data_ptr(), q.data_ptr(), 1, 32769, 1, 4, sel.data_ptr(), None)
    assert rc == SPIN_ERR_INVALID and "32768" in spin.spin_last_error(None)
