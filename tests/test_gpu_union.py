"""GQA with per-query-head selection and a per-KV-head page union (Quest page
§2.1, the MHA / GQA / head-sharing paragraphs): quest_score_pages_per_head
against the oracle's per-head bounds (1e-4 * sum_j |q_j| max(|m_j|, |M_j|)),
per-head selections under the near-tie rule, the union (pages, head bits,
count) bit-exact against the oracle's union of the GPU's own selections, and
quest_union_decode_attn within 2e-3 (row-max-relative) of the oracle's
per-head attention on those selections."""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import (F16, F32, attn_close, check_selection, dev_i32, gpu_cache, gpu_table,
                          np_of, random_case)

pytestmark = pytest.mark.gpu


def _per_head_tol(q, summary, table, group):
    qn = np.abs(np.asarray(q, dtype=np.float64))
    h_q = qn.shape[1]
    tol = np.zeros((h_q, table.nnz))
    for r in range(table.batch):
        lo, hi = int(table.page_indptr[r]), int(table.page_indptr[r + 1])
        phys = table.page_indices[lo:hi]
        mag = np.maximum(np.abs(summary[phys, :, 0].astype(np.float64)),
                         np.abs(summary[phys, :, 1].astype(np.float64)))   # [P, h_kv, d]
        for h in range(h_q):
            tol[h, lo:hi] = 1e-4 * (mag[:, h // group] @ qn[r, h])
    return tol


def _run(seed, lens, h_kv, group, d, S, dtype, k, same_queries=False, drop_heads=False):
    import query_aware_sparse_gb300 as qs
    case = random_case(seed, lens, h_kv=h_kv, group=group, d=d, S=S, dtype=dtype)
    t = case["table"]
    if same_queries:                   # every head of a group asks the same question
        qv = case["q"].view(len(lens), h_kv, group, d)
        case["q"] = qv[:, :, :1].expand(-1, -1, group, -1).contiguous().view(len(lens), -1, d)
    kp, vp = np_of(case["k_pool"]), np_of(case["v_pool"])
    osm = qo.build_summary(kp, t.page_indptr, t.page_indices, t.seq_lens,
                           summary=np_of(case["summary"]).copy())
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(osm))
    table = gpu_table(t)
    q = case["q"]
    qd = q.cuda()
    h_q = h_kv * group
    sc = qs.score_pages_per_head(cache, table, qd, group)
    assert qs.device_error() == 0
    ref = qo.score_pages_per_head(np_of(q), osm, t.page_indptr, t.page_indices, group)
    tol = _per_head_tol(np_of(q), osm, t, group)
    got = np_of(sc)
    for r in range(t.batch):
        lo, hi = int(t.page_indptr[r]), int(t.page_indptr[r + 1])
        P = -(-int(t.seq_lens[r]) // S)
        assert np.all(np.abs(got[:, lo:lo + P] - ref[:, lo:lo + P]) <= tol[:, lo:lo + P])
        assert np.all(got[:, lo + P:hi] == -np.inf)
    sl, sp, cnt = qs.select_topk(table, h_q, S, sc, k)
    sl_np = np_of(sl)
    check_selection(sl_np, np_of(cnt), ref, tol, t, k,
                    [(r, h) for r in range(t.batch) for h in range(h_q)])
    if drop_heads:                      # some heads choose nothing at all
        sl_np = sl_np.copy()
        sl_np[:, 1::3] = -1
        sl = dev_i32(sl_np)
    out, lse, (ul, um, uc) = qs.union_decode_attn(cache, table, qd, group, sl, k)
    assert qs.device_error() == 0
    ul, um, uc = np_of(ul), np_of(um), np_of(uc)
    for r in range(t.batch):
        for g in range(h_kv):
            pages, masks = qo.union_pages(sl_np[r, g * group:(g + 1) * group])
            n = len(pages)
            assert uc[r, g] == n
            assert ul[r, g, :n].tolist() == pages.tolist()
            assert um[r, g, :n].tolist() == masks.tolist()
            assert np.all(ul[r, g, n:] == -1) and np.all(um[r, g, n:] == 0)
            if same_queries:
                assert n == min(k, -(-int(t.seq_lens[r]) // S))
    ro, rl = qo.sparse_attention_per_head(np_of(q), kp, vp, t.page_indptr, t.page_indices,
                                          t.seq_lens, sl_np, group)
    o, l = np_of(out), np_of(lse)
    ok, rel = attn_close(o, ro)
    assert ok.all(), rel.max()
    fin = np.isfinite(rl)
    assert np.allclose(l[fin], rl[fin], rtol=1e-4, atol=1e-4)
    assert np.all(l[~fin] == -np.inf) and np.all(o[~fin] == 0)
    return uc


@pytest.mark.parametrize("group,d,S,dtype", [(4, 128, 16, F16), (2, 64, 32, F16),
                                             (8, 64, 16, F16), (4, 128, 16, F32),
                                             (1, 128, 16, F16)])
def test_union_path_matches_oracle(group, d, S, dtype):
    lens = [1, 15, 16, 17, 250, 1000, 333]
    _run(900 + group + d + S, lens, 2, group, d, S, dtype, k=6)


def test_union_budget_above_pages_and_empty_heads():
    _run(931, [40, 5, 300], 2, 4, 128, 16, F16, k=9, drop_heads=True)


def test_union_of_identical_heads_is_one_set():
    uc = _run(937, [700, 129], 3, 4, 128, 16, F16, k=8, same_queries=True)
    assert np.all(uc == 8)


def test_union_long_rows():
    _run(941, [32768, 9000], 2, 4, 128, 16, F16, k=64)


def test_per_head_scores_over_e4m3_summaries():
    """Per-head rows read E4M3 summaries too: against the oracle's per-head
    bounds over the decoded box (Quest page §3 summary dtype, §2.1 GQA)."""
    import query_aware_sparse_gb300 as qs
    group, S = 4, 16
    case = random_case(951, [1, 17, 500, 2000], h_kv=2, group=group, d=128, S=S, dtype=F16,
                       scale=3.0)
    t = case["table"]
    exact = qo.build_summary(np_of(case["k_pool"]), t.page_indptr, t.page_indices, t.seq_lens)
    codes, ovf = qo.summary_to_e4m3(exact)
    assert not ovf.any()
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(codes))
    q = case["q"]
    got = np_of(qs.score_pages_per_head(cache, gpu_table(t), q.cuda(), group))
    assert qs.device_error() == 0
    box = qo.e4m3_decode(codes)
    ref = qo.score_pages_per_head(np_of(q), box, t.page_indptr, t.page_indices, group)
    tol = _per_head_tol(np_of(q), box, t, group)
    for r in range(t.batch):
        lo = int(t.page_indptr[r])
        P = -(-int(t.seq_lens[r]) // S)
        assert np.all(np.abs(got[:, lo:lo + P] - ref[:, lo:lo + P]) <= tol[:, lo:lo + P])
