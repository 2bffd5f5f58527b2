"""The no-allocation attention entry point (quest_sparse_decode_attn_noalloc).

It is meant for callers that cannot allocate device memory (a plug-in that is
handed only input and output pointers, or a serving loop that must not call
cudaMalloc while running), so it keeps its split-K partials in a fixed buffer
inside the library. These tests call it through the C ABI and compare it with the oracle and with
quest_sparse_decode_attn, which takes a caller-allocated workspace, on two
calls in a row and on a larger problem followed by a smaller one (no call may
depend on what an earlier one left in the shared buffer), and run it at the
largest batch its buffer takes. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import F16, attn_close, dev_i32, gpu_cache, gpu_table, np_of, random_case

pytestmark = pytest.mark.gpu


def _sets(case, k, seed):
    t = case["table"]
    rng = np.random.default_rng(seed)
    sl = np.full((t.batch, case["h_kv"], k), -1, np.int32)
    for r in range(t.batch):
        P = -(-int(t.seq_lens[r]) // t.page_size)
        for g in range(case["h_kv"]):
            n = min(P, k)
            sl[r, g, :n] = np.sort(rng.choice(P, size=n, replace=False)) if n else []
    sp = np.where(sl >= 0, t.page_indices[np.maximum(sl, 0) + t.page_indptr[:-1, None, None]], -1)
    return dev_i32(sl), dev_i32(sp.astype(np.int32))


def _noalloc(cache, table, q, group, sl, sp, k):
    """One call of the C ABI entry point (no workspace argument)."""
    import query_aware_sparse_gb300 as qs
    B, h_q, d = q.shape
    out = torch.full((B, h_q, d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, h_q), float("nan"), dtype=torch.float32, device="cuda")
    st = qs.lib().quest_sparse_decode_attn_noalloc(
        ctypes.byref(cache.c), ctypes.byref(table.c), q.data_ptr(), group, sl.data_ptr(),
        sp.data_ptr(), k, out.data_ptr(), lse.data_ptr(), ctypes.c_float(0.0),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, qs.lib().quest_status_string(st)
    return out, lse


def _check(o, l, ref_o, ref_l, exact=False):
    o, l, ref_o, ref_l = (np.asarray(x) for x in (o, l, ref_o, ref_l))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.all(o[~fin] == 0)
    if exact:                                   # the same kernels on the same plan
        assert np.array_equal(o, ref_o) and np.array_equal(l[fin], ref_l[fin])
        return
    ok, rel = attn_close(o[fin], ref_o[fin])
    assert ok.all(), rel.max()
    assert np.all(np.abs(l[fin] - ref_l[fin]) <= 1e-3 * np.maximum(1, np.abs(ref_l[fin])))


def _oracle(case, sl, group, q):
    t = case["table"]
    return qo.sparse_attention(np_of(q), np_of(case["k_pool"]), np_of(case["v_pool"]),
                               t.page_indptr, t.page_indices, t.seq_lens, np_of(sl), group)


@pytest.mark.parametrize("group,d,S", [(1, 128, 16), (4, 128, 16), (2, 64, 32)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(group, d, S):
    import query_aware_sparse_gb300 as qs
    lens = [1, 17, 0, 300, 2000]
    case = random_case(70 + group, lens, h_kv=2, group=group, d=d, S=S, dtype=F16)
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    table = gpu_table(case["table"])
    k = 24
    sl, sp = _sets(case, k, seed=group)
    q1 = case["q"]
    q2 = (case["q"].float() * -0.5 + 0.25).to(F16)             # a different second query
    for q in (q1, q2):                                          # two calls in a row
        o, l = _noalloc(cache, table, q.cuda(), group, sl, sp, k)
        assert qs.device_error() == 0
        ro, rl = _oracle(case, sl, group, q)
        _check(np_of(o), np_of(l), ro, rl)
        wo, wl_ = qs.sparse_decode_attn(cache, table, q.cuda(), group, sl, sp, k)
        _check(np_of(o), np_of(l), np_of(wo), np_of(wl_), exact=True)


def test_noalloc_larger_problem_then_smaller():
    """A call over more requests leaves more of the shared buffer written; a
    smaller call after it must not read any of that."""
    import query_aware_sparse_gb300 as qs
    k = 32
    big = random_case(81, [900, 40, 5, 1200, 333, 64, 700, 16, 2500], h_kv=4, group=4, d=128,
                      S=16, dtype=F16)
    small = random_case(82, [600, 3], h_kv=4, group=4, d=128, S=16, dtype=F16)
    for case in (big, small):
        cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
        table = gpu_table(case["table"])
        sl, sp = _sets(case, k, seed=5)
        o, l = _noalloc(cache, table, case["q"].cuda(), 4, sl, sp, k)
        assert qs.device_error() == 0
        ro, rl = _oracle(case, sl, 4, case["q"])
        _check(np_of(o), np_of(l), ro, rl)


def test_noalloc_near_its_buffer_limit():
    """The largest batch whose partials still fit the 4 MiB buffer (sized by
    quest_attn_workspace_size, which covers both element types) runs, and
    equals the workspace entry point; sampled requests match the oracle."""
    import query_aware_sparse_gb300 as qs
    h_kv, G, d, S, k = 8, 8, 128, 16, 64
    B = 1
    while qs.attn_workspace_size(B + 1, h_kv, G, d, S, k) <= (4 << 20) and B < 4096:
        B += 1
    need = qs.attn_workspace_size(B, h_kv, G, d, S, k)
    assert (3 << 20) < need <= (4 << 20), (B, need)
    rng = np.random.default_rng(83)
    lens = [int(x) for x in rng.integers(1, 48 * S, B)]
    case = random_case(84, lens, h_kv=h_kv, group=G, d=d, S=S, dtype=F16, spare=0)
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    table = gpu_table(case["table"])
    sl, sp = _sets(case, k, seed=6)
    q = case["q"].cuda()
    o, l = _noalloc(cache, table, q, G, sl, sp, k)
    assert qs.device_error() == 0
    wo, wl_ = qs.sparse_decode_attn(cache, table, q, G, sl, sp, k)
    _check(np_of(o), np_of(l), np_of(wo), np_of(wl_), exact=True)
    pick = np.sort(rng.choice(B, size=min(B, 6), replace=False))
    t = case["table"]
    ro, rl = qo.sparse_attention(np_of(case["q"]), np_of(case["k_pool"]), np_of(case["v_pool"]),
                                 t.page_indptr, t.page_indices, t.seq_lens, np_of(sl), G,
                                 requests=pick)
    _check(np_of(o)[pick], np_of(l)[pick], ro[pick], rl[pick])


def test_noalloc_rejects_problems_beyond_its_buffer():
    import query_aware_sparse_gb300 as qs
    # 64 requests x 64 KV heads x 8 query heads with K = 4096 needs far more
    # than 4 MiB of split-K partials; the call must refuse before launching
    B, h_kv, G, d, k = 64, 64, 8, 128, 4096
    need = qs.attn_workspace_size(B, h_kv, G, d, 16, k)
    assert need > (4 << 20)
    kp = torch.zeros((1, h_kv, 16, d), dtype=F16, device="cuda")
    cache = qs.PagedCache(kp, kp, torch.zeros((1, h_kv, 2, d), dtype=F16, device="cuda"))
    table = qs.PageTable(dev_i32(np.zeros(B + 1)), dev_i32([0]), dev_i32(np.zeros(B)), nnz=0)
    q = torch.zeros((B, h_kv * G, d), dtype=F16, device="cuda")
    sel = torch.full((B, h_kv, k), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, h_kv * G, d), dtype=torch.float32, device="cuda")
    st = qs.lib().quest_sparse_decode_attn_noalloc(
        ctypes.byref(cache.c), ctypes.byref(table.c), q.data_ptr(), G, sel.data_ptr(),
        sel.data_ptr(), k, out.data_ptr(), None, ctypes.c_float(0.0), None)
    assert st == -3, qs.lib().quest_status_string(st)
