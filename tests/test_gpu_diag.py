"""f4 parity: quest_recall_diagnostics against the oracle's fp64
recall_diagnostics (Quest page §1.1 recall paragraph, eq (6)-(7); §3.1 page
slack) on the same stored inputs and the same selection.

Tolerances: slack within 1e-5 * sum_j |q_j| max(|m_j|, |M_j|) (fp32 dot
products and page bound against fp64); eps within 1e-5 absolute (fp32 sums
of at most a few thousand terms of [0, 1]); V_max within 1e-5 relative; the
top-R recall exactly, except that tokens whose dense logit lies within the
logit tolerance of the R-th logit may swap places (the fp32 and fp64 orders
can differ there), so the hit counts may differ by at most their number.
"""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import F16, F32, dev_i32, gpu_cache, gpu_table, np_of, random_case

pytestmark = pytest.mark.gpu


def _selection(rng, table, h_kv, k):
    """Random selections: some full, some partial, some empty, -1 padded."""
    B = table.batch
    sel = np.full((B, h_kv, k), -1, np.int32)
    for r in range(B):
        P = -(-int(table.seq_lens[r]) // table.page_size)
        for g in range(h_kv):
            n = int(rng.integers(0, min(P, k) + 1))
            chosen = rng.choice(P, size=n, replace=False)
            sel[r, g, :n] = rng.permutation(chosen)
    return sel


def _run(seed, lens, h_kv, group, d, S, dtype, k, R):
    import query_aware_sparse_gb300 as qs
    case = random_case(seed, lens, h_kv=h_kv, group=group, d=d, S=S, dtype=dtype)
    t = case["table"]
    kp, vp = np_of(case["k_pool"]), np_of(case["v_pool"])
    osm = qo.build_summary(kp, t.page_indptr, t.page_indices, t.seq_lens,
                           summary=np_of(case["summary"]).copy())
    sel = _selection(np.random.default_rng(seed), t, h_kv, k)
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(osm))
    q = case["q"]
    got = qs.recall_diagnostics(cache, gpu_table(t), q.cuda(), group, dev_i32(sel), k, R)
    assert qs.device_error() == 0
    got = {n: np_of(v) for n, v in got.items()}
    ref = qo.recall_diagnostics(np_of(q), kp, vp, t.page_indptr, t.page_indices, t.seq_lens,
                                sel, group, R)
    qn = np.abs(np_of(q).astype(np.float64))
    # slack
    for r in range(t.batch):
        lo, hi = int(t.page_indptr[r]), int(t.page_indptr[r + 1])
        P = -(-int(t.seq_lens[r]) // S)
        for h in range(h_kv * group):
            g = h // group
            for lp in range(P):
                pp = t.page_indices[lo + lp]
                mag = np.maximum(np.abs(osm[pp, g, 0].astype(np.float64)),
                                 np.abs(osm[pp, g, 1].astype(np.float64)))
                tol = 1e-5 * float(mag @ qn[r, h]) + 1e-6
                assert abs(got["slack"][h, lo + lp] - ref["slack"][h, lo + lp]) <= tol
            assert np.all(np.isnan(got["slack"][:, lo + P:hi]))
    assert np.all(got["slack"][~np.isnan(ref["slack"])] >= -1e-3)
    # eps and V_max
    assert np.all(np.abs(got["eps"] - ref["eps"]) <= 1e-5), np.max(np.abs(got["eps"] - ref["eps"]))
    assert np.allclose(got["vmax"], ref["vmax"], rtol=1e-5, atol=0)
    # top-R recall, with the near-tie allowance
    for r in range(t.batch):
        L = int(t.seq_lens[r])
        Rr = min(R, L)
        for h in range(h_kv * group):
            g = h // group
            keys, _ = qo.candidate_tokens(kp, vp, t.page_indptr, t.page_indices, t.seq_lens, r,
                                          g, range(-(-L // S)))
            s = keys @ np_of(q)[r, h].astype(np.float64)
            tau = np.sort(s)[::-1][Rr - 1]
            stol = 1e-5 * float(np.abs(keys).max(axis=0) @ qn[r, h]) + 1e-6
            amb = int(np.sum(np.abs(s - tau) <= stol))
            diff = abs(round(got["topr"][r, h] * Rr) - round(ref["topr"][r, h] * Rr))
            assert diff <= (amb if amb > 1 else 0), (r, h, got["topr"][r, h], ref["topr"][r, h])
    return got, ref, case, sel


@pytest.mark.parametrize("dtype,d,S,group", [(F16, 64, 16, 1), (F16, 128, 16, 4),
                                             (F32, 64, 32, 2), (F16, 128, 32, 8)])
def test_diagnostics_match_oracle(dtype, d, S, group):
    _run(40 + d + S + group, [1000, 37, 1, 16, 300], h_kv=2, group=group, d=d, S=S,
         dtype=dtype, k=8, R=20)


def test_diagnostics_bound_eq7_on_gpu_attention():
    """||o_dense - o_C|| <= 2 eps V_max with o_C from quest_sparse_decode_attn
    and eps, V_max from the GPU diagnostics (Quest page eq (7))."""
    import query_aware_sparse_gb300 as qs
    got, ref, case, sel = _run(77, [700, 90], h_kv=2, group=2, d=64, S=16, dtype=F16, k=6, R=8)
    t = case["table"]
    kp, vp = np_of(case["k_pool"]), np_of(case["v_pool"])
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    phys = np.where(sel >= 0, t.page_indices[t.page_indptr[:-1, None, None] + np.maximum(sel, 0)], -1)
    o, _ = qs.sparse_decode_attn(cache, gpu_table(t), case["q"].cuda(), 2, dev_i32(sel),
                                 dev_i32(phys.astype(np.int32)), 6)
    o = np_of(o)
    for r in range(t.batch):
        L = int(t.seq_lens[r])
        for h in range(4):
            g = h // 2
            keys, vals = qo.candidate_tokens(kp, vp, t.page_indptr, t.page_indices, t.seq_lens,
                                             r, g, range(-(-L // 16)))
            od, _ = qo.dense_attention(np_of(case["q"])[r, h], keys, vals)
            bound = 2 * got["eps"][r, h] * got["vmax"][r, g]
            assert np.linalg.norm(od - o[r, h]) <= bound + 2e-3 * max(1.0, np.abs(od).max())


def test_diagnostics_top_r_above_length_and_full_selection():
    import query_aware_sparse_gb300 as qs
    lens = [5, 40]
    case = random_case(91, lens, h_kv=1, group=1, d=64, S=16, dtype=F16)
    t = case["table"]
    osm = qo.build_summary(np_of(case["k_pool"]), t.page_indptr, t.page_indices, t.seq_lens,
                           summary=np_of(case["summary"]).copy())
    sel = np.full((2, 1, 4), -1, np.int32)
    sel[0, 0, 0] = 0
    sel[1, 0, :3] = [2, 0, 1]
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(osm))
    got = qs.recall_diagnostics(cache, gpu_table(t), case["q"].cuda(), 1, dev_i32(sel), 4, 1000)
    assert qs.device_error() == 0
    assert np.all(np_of(got["eps"]) == 0) and np.all(np_of(got["topr"]) == 1)
