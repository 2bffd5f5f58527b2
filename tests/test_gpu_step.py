"""Fused decode step (quest_decode_step): every output against the oracle's
chain on the same inputs — summaries and pool bit-exact, scores within the
score tolerance, selections under the near-tie rule, attention within 2e-3 —
over several consecutive steps (the workspace counters must come back to
zero), with and without the append, MHA and GQA, page sizes 16 and 32."""

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quest_oracle as qo
from tests._cases import (attn_close, check_selection, dev_i32, gpu_table, np_of,
                          score_tol)

pytestmark = pytest.mark.gpu


def _prefilled(w, lens, seed, spare=4):
    """Pools holding every token but the last of each request (host+device),
    and the tokens themselves."""
    import query_aware_sparse_gb300 as qs
    table = wl.make_page_table(lens, w.page_size, seed=seed, permute=True,
                               spare_pages=spare, reserve_tokens=2 * w.page_size)
    k_tok, v_tok, ind = wl.tokens_for_table(w, table)
    return table, k_tok, v_tok, ind


def _run(w, lens, steps, seed, append=True, n_sink=0, n_local=0, fp8=False):
    import query_aware_sparse_gb300 as qs
    lens = np.asarray(lens)
    full = lens + (steps if append else 0)
    table, k_tok, v_tok, ind = _prefilled(w, full, seed)
    h, d, S, B = w.h_kv, w.head_dim, w.page_size, len(lens)
    start = lens.copy()
    # both sides start from the first `lens` tokens of each request
    kp, vp, sm = wl.empty_pool(table, h, d, w.dtype, device="cuda")
    if fp8:                                  # E4M3 summary codes instead
        sm = torch.full(sm.shape, 0x7F, dtype=torch.uint8, device="cuda")
    okp, ovp, osm = (np_of(x) for x in wl.empty_pool(table, h, d, w.dtype))
    rows = np.concatenate([np.arange(ind[r], ind[r] + start[r]) for r in range(B)])
    pre_ind = np.concatenate([[0], np.cumsum(start)]).astype(np.int32)
    kn, vn = k_tok[rows].contiguous(), v_tok[rows].contiguous()
    cache = qs.PagedCache(kp, vp, sm)
    gt = gpu_table(table, seq_lens=start.astype(np.int32))
    qs.append_kv(cache, gt, kn.cuda(), vn.cuda(), dev_i32(pre_ind), dev_i32(np.zeros(B)))
    qo.append_kv(okp, ovp, osm, table.page_indptr, table.page_indices, np.zeros(B, np.int32),
                 pre_ind, np_of(kn), np_of(vn))
    step = None
    cur = start.copy()
    for s in range(steps):
        if append:
            cur = cur + 1
            pos = ind[:-1] + cur - 1
            k1, v1 = k_tok[pos].contiguous(), v_tok[pos].contiguous()
        q = wl.queries(w, cur - 1, step=s)
        tb = wl.PageTable(table.page_indptr, table.page_indices, cur.astype(np.int32),
                          table.n_phys, S)
        gtab = gpu_table(tb)
        if step is None:
            step = qs.DecodeStep(cache, gtab, w.group, w.k, n_sink=n_sink, n_local=n_local)
        if append:
            step(cache, gtab, q.cuda(), k1.cuda(), v1.cuda())
            qo.append_kv(okp, ovp, osm, table.page_indptr, table.page_indices,
                         (cur - 1).astype(np.int32), np.arange(B + 1), np_of(k1), np_of(v1))
        else:
            step(cache, gtab, q.cuda())
        assert qs.device_error() == 0
        if step.workspace.numel() > 256:
            # the grid-wide kernel: after every call the call tag and the
            # ready flags hold the number of calls made so far, the per-unit
            # slot counters are back at zero, this call's counted-in bank (tag
            # parity) holds every CTA and the next call's bank is clear (the
            # cluster kernel uses no workspace)
            cnt = step.workspace[:(4 + 2 * B * h) * 4].view(torch.int32).cpu().numpy()
            assert cnt[0] == s + 1 and cnt[1] == 0
            assert cnt[2 + ((s + 1) & 1)] > 0 and cnt[2 + ((s + 2) & 1)] == 0
            assert np.all(cnt[4:4 + B * h] == s + 1) and np.all(cnt[4 + B * h:] == 0)
        gsm = np_of(cache.summary)
        # the summary the selector reads: exact, or its E4M3 rounding
        ssm = qo.summary_to_e4m3(osm)[0] if fp8 else osm
        for r in range(B):
            P = -(-int(cur[r]) // S)
            phys = table.page_indices[table.page_indptr[r]:table.page_indptr[r] + P]
            assert np.array_equal(gsm[phys].view(np.uint8), ssm[phys].view(np.uint8))
            if append:
                pp = table.page_indices[table.page_indptr[r] + (cur[r] - 1) // S]
                slot = (cur[r] - 1) % S
                assert np.array_equal(np_of(cache.k_pool[pp, :, slot]).view(np.uint8),
                                      okp[pp, :, slot].view(np.uint8))
        if fp8:
            ref_scores = qo.score_pages_e4m3(np_of(q), ssm, table.page_indptr, table.page_indices,
                                             w.group)
            tol = score_tol(np_of(q), qo.e4m3_decode(ssm), tb, w.group)
        else:
            ref_scores = qo.score_pages(np_of(q), osm, table.page_indptr, table.page_indices, w.group)
            tol = score_tol(np_of(q), osm, tb, w.group)
        got = np_of(step.scores)
        for r in range(B):
            lo = table.page_indptr[r]
            P = -(-int(cur[r]) // S)
            assert np.all(np.abs(got[:, lo:lo + P] - ref_scores[:, lo:lo + P]) <= tol[:, lo:lo + P])
            assert np.all(got[:, lo + P:table.page_indptr[r + 1]] == -np.inf)
        sl, sp, cnt = (np_of(x) for x in step.sel)
        check_selection(sl, cnt, ref_scores, tol, tb, w.k,
                        [(r, g) for r in range(B) for g in range(h)], n_sink, n_local)
        ref_sel, _, _ = qo.select_hybrid(np.where(np.isfinite(ref_scores), ref_scores, -np.inf),
                                         table.page_indptr, table.page_indices, cur, S, w.k,
                                         n_sink, n_local)
        assert np.array_equal(sp[sl >= 0], table.page_indices[(table.page_indptr[:-1, None, None] + sl)[sl >= 0]])
        use = ref_sel if np.array_equal(sl, ref_sel) else sl
        ro, rl = qo.sparse_attention(np_of(q), okp, ovp, table.page_indptr, table.page_indices,
                                     cur.astype(np.int32), use, w.group)
        o, lse = np_of(step.out), np_of(step.lse)
        ok, rel = attn_close(o, ro)
        assert ok.all(), rel.max()
        fin = np.isfinite(rl)
        assert np.allclose(lse[fin], rl[fin], rtol=1e-4, atol=1e-4)
        assert np.all(lse[~fin] == -np.inf) and np.all(o[~fin] == 0)


def _w(name, **kw):
    base = dict(batch=1, h_kv=4, group=1, head_dim=128, page_size=16, k=16,
                dtype=torch.float16, seed=500)
    base.update(kw)
    return wl.Workload(name, **base)


@pytest.fixture(params=["cluster", "grid"])
def kernel(request, monkeypatch):
    """The cluster kernel runs groups 1 and 2 (and 4 and 8 with fp16 K/V);
    QUEST_STEP_LEGACY selects the grid-wide kernel instead."""
    if request.param == "grid":
        monkeypatch.setenv("QUEST_STEP_LEGACY", "1")
    return request.param


def test_step_mha_crosses_page_boundaries(kernel):
    # 30 -> 31, 32 (page full), 33 (fresh page: slot 0), 34
    _run(_w("mha", batch=3, h_kv=4), [30, 1, 200], steps=4, seed=1)


@pytest.mark.parametrize("group", [2, 4, 8])
def test_step_gqa_ragged(group, kernel):
    _run(_w("gqa", batch=5, h_kv=2, group=group, k=24), [1, 15, 16, 17, 900], steps=2,
         seed=2 + group)


def test_step_page32_fp16():
    _run(_w("p32", batch=2, h_kv=3, page_size=32, k=8), [31, 500], steps=3, seed=7)


@pytest.mark.parametrize("group,S,d", [(4, 32, 64), (8, 32, 128), (4, 16, 64), (8, 32, 64)])
def test_step_gqa_tiles(group, S, d, kernel):
    """Groups of 4 and 8 over every page size and head dim: sub-blocks of one
    and of two 16-token attention tiles, ragged last pages."""
    _run(_w("gqa_t", batch=3, h_kv=2, group=group, head_dim=d, page_size=S, k=12),
         [S + 3, 7 * S - 5, 40 * S + 1], steps=2, seed=30 + group + S + d)


def test_step_fp32_d64():
    _run(_w("f32", batch=2, h_kv=2, head_dim=64, dtype=torch.float32, k=8), [1000, 63],
         steps=2, seed=8)


def test_step_without_append_and_k_above_pages():
    _run(_w("noapp", batch=3, h_kv=2, k=40), [100, 700, 5], steps=2, seed=9, append=False)


def test_step_many_units(kernel):
    # more (request, head) units than select workers and CTAs per head
    _run(_w("many", batch=24, h_kv=8, group=1, k=8, head_dim=64), list(range(10, 250, 10)),
         steps=1, seed=10)


def test_step_units_above_grid(kernel):
    # more units than CTAs (one per SM at G = 4): CTAs select several units
    # each after scoring
    _run(_w("above", batch=20, h_kv=8, group=4, k=4, head_dim=64),
         [17 + 13 * i for i in range(20)], steps=2, seed=11)


@pytest.mark.parametrize("group,lens", [(1, [70000, 900]), (1, [140000, 3000]),
                                        (4, [140000, 3000])])
def test_step_long_rows(group, lens, kernel):
    # rows above the 4096 and 8192 keys the selecting CTA caches in shared
    # memory (the second reads its keys from L2)
    _run(_w("long", batch=2, h_kv=2, group=group, k=64, head_dim=64), lens, steps=2,
         seed=12 + group)


def test_step_fp32_d128_gqa():
    _run(_w("f32g", batch=3, h_kv=2, group=2, head_dim=128, dtype=torch.float32, k=8),
         [300, 17, 1000], steps=2, seed=13)


@pytest.mark.parametrize("n_sink,n_local", [(1, 4), (2, 0), (0, 16)])
def test_step_hybrid_budget(n_sink, n_local):
    """Local window + sink pages forced (Quest page §2.2, §3.2), through the
    fused step, with short requests whose window and sinks overlap."""
    _run(_w("hyb", batch=4, h_kv=3, k=16), [40, 1, 300, 700], steps=3, seed=20 + n_local,
         n_sink=n_sink, n_local=n_local)


@pytest.mark.parametrize("group,S,d", [(1, 16, 128), (4, 16, 128), (2, 32, 64), (8, 16, 64),
                                       (1, 32, 128)])
def test_step_e4m3_summaries(group, S, d, kernel):
    """E4M3 summaries (Quest page §3, summary dtype): the fused append keeps
    the codes equal to the directed rounding of the exact summary, and the
    scores, selections and outputs follow the oracle on the rounded box."""
    w = _w("e4m3", batch=3, h_kv=2, group=group, head_dim=d, page_size=S, k=6)
    _run(w, [S - 2, 5 * S, 3 * S + 7], 4, 640 + group + S + d, fp8=True)


def test_step_e4m3_hybrid_and_many_units():
    w = _w("e4m3_units", batch=24, h_kv=8, group=1, k=8)
    _run(w, list(np.random.default_rng(3).integers(20, 400, 24)), 3, 661, n_sink=1, n_local=2,
         fp8=True)
