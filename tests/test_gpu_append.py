"""a1 parity: quest_append_kv against the oracle's eq (8) append, bit-exact
(pool contents and min/max summaries, signed zeros included)."""

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quest_oracle as qo
from tests._cases import F16, F32, dev_i32, gpu_table, np_of, random_case

pytestmark = pytest.mark.gpu


def _run_appends(case, chunks):
    """Append the case's tokens in the given per-request chunk schedule on both
    sides. chunks: list of lists, chunks[step][r] = tokens of request r."""
    import query_aware_sparse_gb300 as qs
    t = case["table"]
    kp, vp, sm = (x.clone() for x in (case["k_pool"], case["v_pool"], case["summary"]))
    # both sides start from the same NaN-poisoned pool, never from the
    # case's pre-placed tokens
    kp[:] = float("nan"); vp[:] = float("nan"); sm[:] = float("nan")
    okp, ovp, osm = np_of(kp), np_of(vp), np_of(sm)
    cache = qs.PagedCache(kp.cuda(), vp.cuda(), sm.cuda())
    done = np.zeros(t.batch, dtype=np.int64)
    starts = case["tok_indptr"]
    for step in chunks:
        rows, ind = [], [0]
        for r, n in enumerate(step):
            a = starts[r] + done[r]
            rows.append(np.arange(a, a + n))
            ind.append(ind[-1] + n)
        rows = np.concatenate(rows).astype(np.int64)
        kn = case["k_tok"][rows].contiguous()
        vn = case["v_tok"][rows].contiguous()
        before = done.astype(np.int32)
        qo.append_kv(okp, ovp, osm, t.page_indptr, t.page_indices, before,
                     np.asarray(ind), np_of(kn), np_of(vn))
        table = gpu_table(t, seq_lens=(done + np.asarray(step)).astype(np.int32))
        qs.append_kv(cache, table, kn.cuda(), vn.cuda(), dev_i32(ind), dev_i32(before))
        done += np.asarray(step)
    assert qs.device_error() == 0
    return cache, (okp, ovp, osm)


def _bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint16 if a.dtype == np.float16 else np.uint32)


def _assert_same(cache, ref, table):
    okp, ovp, osm = ref
    gk, gv, gs = np_of(cache.k_pool), np_of(cache.v_pool), np_of(cache.summary)
    S = table.page_size
    for r in range(table.batch):
        L = int(table.seq_lens[r])
        for p in range(-(-L // S)):
            pp = table.page_indices[table.page_indptr[r] + p]
            valid = min(S, L - p * S)
            assert np.array_equal(_bits(gs[pp]), _bits(osm[pp])), (r, p)
            assert np.array_equal(_bits(gk[pp, :, :valid]), _bits(okp[pp, :, :valid]))
            assert np.array_equal(_bits(gv[pp, :, :valid]), _bits(ovp[pp, :, :valid]))


@pytest.mark.parametrize("dtype,d,S", [(F16, 128, 16), (F16, 64, 32), (F32, 64, 16),
                                       (F32, 128, 32), (F16, 128, 32)])
def test_prefill_tail_lengths(dtype, d, S):
    lens = [1, 15, 16, 17, S - 1, S + 1, 3 * S, 100]
    case = random_case(3, lens, h_kv=3, d=d, S=S, dtype=dtype, signed_zeros=True)
    cache, ref = _run_appends(case, [lens])
    _assert_same(cache, ref, case["table"])


def test_decode_appends_one_token_at_a_time():
    lens = [1, 16, 17, 40]
    case = random_case(5, lens, h_kv=2, d=128, S=16, signed_zeros=True)
    sched = []
    done = [0] * len(lens)
    while any(d < L for d, L in zip(done, lens)):
        step = [1 if d < L else 0 for d, L in zip(done, lens)]
        sched.append(step)
        done = [d + s for d, s in zip(done, step)]
    cache, ref = _run_appends(case, sched)
    _assert_same(cache, ref, case["table"])


def test_mixed_chunked_prefill():
    lens = [50, 7, 33, 64, 0, 21]
    case = random_case(7, lens, h_kv=4, d=64, S=16, dtype=F32, signed_zeros=True)
    sched = [[10, 3, 17, 16, 0, 1], [25, 4, 0, 16, 0, 19], [15, 0, 16, 32, 0, 1]]
    cache, ref = _run_appends(case, sched)
    _assert_same(cache, ref, case["table"])


def test_slot_reuse_restarts_summary():
    """Fill a physical page for one request, then hand it to another request
    with fewer tokens: its summary must equal a fresh page's (page recycling)."""
    import query_aware_sparse_gb300 as qs
    S, d, h = 16, 128, 2
    g = torch.Generator().manual_seed(11)
    old = (torch.randn((S, h, d), generator=g) * 10).half()
    new = torch.randn((5, h, d), generator=g).half()
    kp = torch.zeros((1, h, S, d), dtype=F16, device="cuda")
    cache = qs.PagedCache(kp, torch.zeros_like(kp), torch.zeros((1, h, 2, d), dtype=F16, device="cuda"))
    one = qs.PageTable(dev_i32([0, 1]), dev_i32([0]), dev_i32([S]))
    qs.append_kv(cache, one, old.cuda(), old.cuda(), dev_i32([0, S]), dev_i32([0]))
    qs.append_kv(cache, one, new.cuda(), new.cuda(), dev_i32([0, 5]), dev_i32([0]))
    fresh_s = np.zeros((1, h, 2, d), np.float16)
    qo.append_kv(np.zeros((1, h, S, d), np.float16), np.zeros((1, h, S, d), np.float16),
                 fresh_s, np.array([0, 1]), np.array([0]), np.array([0]),
                 np.array([0, 5]), np_of(new), np_of(new))
    assert np.array_equal(np_of(cache.summary), fresh_s)
    assert qs.device_error() == 0


def test_append_beyond_table_is_reported_not_written():
    import query_aware_sparse_gb300 as qs
    S, d, h = 16, 64, 1
    kp = torch.zeros((2, h, S, d), dtype=F16, device="cuda")
    cache = qs.PagedCache(kp, torch.zeros_like(kp), torch.zeros((2, h, 2, d), dtype=F16, device="cuda"))
    table = qs.PageTable(dev_i32([0, 1]), dev_i32([0]), dev_i32([20]))
    k = torch.ones((20, h, d), dtype=F16, device="cuda")
    qs.append_kv(cache, table, k, k, dev_i32([0, 20]), dev_i32([0]))
    assert qs.device_error() & 2
    assert torch.all(cache.k_pool[1] == 0)          # the unmapped page is untouched
