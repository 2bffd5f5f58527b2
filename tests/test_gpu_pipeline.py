"""The whole hot path on small cases: append -> score -> select -> attention
through the C ABI, each step checked against the oracle's own chain."""

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quest_oracle as qo
from tests._cases import (attn_close, check_selection, dev_i32, gpu_table, np_of,
                          score_tol)

pytestmark = pytest.mark.gpu


def run_chain(w: wl.Workload, table: wl.PageTable, k_tok, v_tok, tok_indptr, q, k):
    """GPU chain and oracle chain on the same stored inputs; returns both."""
    import query_aware_sparse_gb300 as qs
    h, d, S = w.h_kv, w.head_dim, w.page_size
    kp, vp, sm = wl.empty_pool(table, h, d, w.dtype, device="cuda")
    cache = qs.PagedCache(kp, vp, sm)
    gt = gpu_table(table)
    zeros = dev_i32(np.zeros(table.batch))
    qs.append_kv(cache, gt, k_tok.cuda(), v_tok.cuda(), dev_i32(tok_indptr), zeros)
    scores = qs.score_pages(cache, gt, q.cuda(), w.group)
    sl, sp, cnt = qs.select_topk(gt, h, S, scores, k)
    o, lse = qs.sparse_decode_attn(cache, gt, q.cuda(), w.group, sl, sp, k)
    assert qs.device_error() == 0

    okp, ovp, osm = (np_of(x) for x in wl.empty_pool(table, h, d, w.dtype))
    qo.append_kv(okp, ovp, osm, table.page_indptr, table.page_indices,
                 np.zeros(table.batch, np.int32), tok_indptr, np_of(k_tok), np_of(v_tok))
    ref_scores = qo.score_pages(np_of(q), osm, table.page_indptr, table.page_indices, w.group)
    ref_sel, _, _ = qo.select_topk(ref_scores, table.page_indptr, table.page_indices, k)
    return dict(cache=cache, scores=np_of(scores), sel=np_of(sl), phys=np_of(sp), cnt=np_of(cnt),
                o=np_of(o), lse=np_of(lse), okp=okp, ovp=ovp, osm=osm, ref_scores=ref_scores,
                ref_sel=ref_sel)


def check_chain(res, table, q, w, k):
    gsm = np_of(res["cache"].summary)
    for r in range(table.batch):
        P = -(-int(table.seq_lens[r]) // table.page_size)
        phys = table.page_indices[table.page_indptr[r]:table.page_indptr[r] + P]
        assert np.array_equal(gsm[phys].view(np.uint8), res["osm"][phys].view(np.uint8))
    tol = score_tol(np_of(q), res["osm"], table, w.group)
    live = np.isfinite(res["ref_scores"])
    assert np.all(np.abs(res["scores"][live] - res["ref_scores"][live]) <= tol[live])
    rows = [(r, g) for r in range(table.batch) for g in range(w.h_kv)]
    check_selection(res["sel"], res["cnt"], res["ref_scores"], tol, table, k, rows)
    # attention: on the oracle's set when the GPU picked the same one, else on
    # the GPU's set, which check_selection has just shown to be a valid choice
    same = np.array_equal(res["sel"], res["ref_sel"])
    use = res["ref_sel"] if same else res["sel"]
    ro, rl = qo.sparse_attention(np_of(q), res["okp"], res["ovp"], table.page_indptr,
                                 table.page_indices, table.seq_lens, use, w.group)
    ok, rel = attn_close(res["o"], ro)
    assert ok.all(), rel.max()
    assert np.allclose(res["lse"], rl, rtol=1e-4, atol=1e-4)
    return same


def test_tiny_workload_end_to_end():
    w = wl.WORKLOADS["tiny"]
    table = wl.make_page_table(w.lengths(), w.page_size, seed=w.seed)
    assert table.nnz == 63 and int(table.seq_lens[0]) - 62 * 16 == 8
    k_tok, v_tok, ind = wl.tokens_for_table(w, table)
    q = wl.queries(w, table.seq_lens - 1)
    res = run_chain(w, table, k_tok, v_tok, ind, q, w.k)
    check_chain(res, table, q, w, w.k)


@pytest.mark.parametrize("group", [1, 4])
def test_ragged_batch_end_to_end(group):
    w = wl.Workload("ragged", batch=5, h_kv=2, group=group, head_dim=128, page_size=16,
                    k=16, dtype=torch.float16, seed=77, seq_lens=(1, 255, 256, 257, 2000))
    table = wl.make_page_table(w.lengths(), 16, seed=w.seed, permute=True, spare_pages=9)
    k_tok, v_tok, ind = wl.tokens_for_table(w, table)
    q = wl.queries(w, table.seq_lens - 1)
    res = run_chain(w, table, k_tok, v_tok, ind, q, w.k)
    check_chain(res, table, q, w, w.k)


def test_fig2_two_step_embedded(golden):
    """Quest page Fig. 2 in d=64 / S=16: page A's three keys repeated to fill
    its 16 slots (repeats change no min/max), page B with two keys, then the
    decode append of (-2, 5); K = 1 moves from A to B."""
    import query_aware_sparse_gb300 as qs
    ex = golden("fig2_two_step.json")
    pr = ex["printed"]
    d, S = 64, 16
    A = np.array(ex["A_keys"], np.float32)
    B = np.array(ex["B_keys_before"], np.float32)
    toks = np.zeros((18, 1, d), np.float32)
    toks[:16, 0, :2] = A[np.arange(16) % 3]
    toks[16:, 0, :2] = B
    kp = torch.full((2, 1, S, d), float("nan"), device="cuda")
    cache = qs.PagedCache(kp, kp.clone(), torch.zeros((2, 1, 2, d), device="cuda"))
    table = qs.PageTable(dev_i32([0, 2]), dev_i32([1, 0]), dev_i32([18]))
    t = torch.from_numpy(toks).cuda()
    qs.append_kv(cache, table, t, t, dev_i32([0, 18]), dev_i32([0]))

    def qv(x):
        q = torch.zeros((1, 1, d), device="cuda")
        q[0, 0, :2] = torch.tensor(x, dtype=torch.float32)
        return q

    sc = np_of(qs.score_pages(cache, table, qv(ex["q_t"]), 1))[0]
    assert sc.tolist() == [pr["U_A_qt"], pr["U_B_qt"]]
    sl, _, _ = qs.select_topk(table, 1, S, torch.from_numpy(sc[None]).cuda(), 1)
    assert np_of(sl)[0, 0, 0] == 0
    assert np_of(qs.score_pages(cache, table, qv(ex["q_t1"]), 1))[0, 1] == pr["U_B_qt1_without_append"]
    new = torch.zeros((1, 1, d), device="cuda")
    new[0, 0, :2] = torch.tensor(ex["appended_key"], dtype=torch.float32)
    table = qs.PageTable(dev_i32([0, 2]), dev_i32([1, 0]), dev_i32([19]))
    qs.append_kv(cache, table, new, new, dev_i32([0, 1]), dev_i32([18]))
    smB = np_of(cache.summary)[0, 0]
    assert smB[0, :2].tolist() == pr["m_B_after"] and smB[1, :2].tolist() == pr["M_B_after"]
    sc = np_of(qs.score_pages(cache, table, qv(ex["q_t1"]), 1))[0]
    assert sc.tolist() == [pr["U_A_qt1"], pr["U_B_qt1"]]
    sl, sp, _ = qs.select_topk(table, 1, S, torch.from_numpy(sc[None]).cuda(), 1)
    assert np_of(sl)[0, 0, 0] == 1 and np_of(sp)[0, 0, 0] == 0
    assert qs.device_error() == 0
