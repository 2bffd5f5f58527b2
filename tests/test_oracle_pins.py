"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here needs a GPU. Each test checks the oracle against a value the
pages print, a closed form, a library routine or brute force, chosen so that
a plausible slip (dropped term, wrong sign, transposed operand, wrong tie
rule, padding leaking into a page) fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo


def _np(x, dt=np.float64):
    return np.asarray(x, dtype=dt)


# --------------------------------------------------------------------------
# Worked examples printed on the Quest page
# --------------------------------------------------------------------------

def test_worked_example_2d(golden):
    ex = golden("worked_example_2d.json")
    for dt in (np.float16, np.float32):
        keys = _np(ex["page"]["keys"], dt)
        m, M = qo.page_summary(keys)
        assert m.tolist() == ex["page"]["m"]
        assert M.tolist() == ex["page"]["M"]
        q = _np(ex["q"])
        assert qo.page_bound(q, m, M) == ex["U"]
        assert (keys.astype(np.float64) @ q).tolist() == ex["dots"]
        # eq (5): the bound equals the page's true maximum here
        assert max(ex["dots"]) == ex["U"]


def test_worked_example_swapped_keys(golden):
    sw = golden("worked_example_2d.json")["swapped"]
    keys = _np(sw["keys"], np.float32)
    m, M = qo.page_summary(keys)
    assert m.tolist() == sw["m"] and M.tolist() == sw["M"]
    q = _np(golden("worked_example_2d.json")["q"])
    assert qo.page_bound(q, m, M) == sw["U"]
    assert (keys.astype(np.float64) @ q).tolist() == sw["dots"]
    assert qo.page_slack(q, keys) == sw["slack"]


def _fig2_state(ex, with_append):
    S = ex["page_size"]
    A = _np(ex["A_keys"], np.float32)
    B = _np(ex["B_keys_before"], np.float32)
    toks = np.concatenate([A, B])[:, None, :]             # [5, h_kv=1, d=2]
    pool_shape = (2, 1, S, 2)
    k_pool = np.full(pool_shape, np.nan, np.float32)
    v_pool = np.full(pool_shape, np.nan, np.float32)
    summ = np.full((2, 1, 2, 2), np.nan, np.float32)
    # two requests' worth of pages is not needed: one request, pages A then B
    indptr = np.array([0, 2], np.int32)
    indices = np.array([0, 1], np.int32)
    qo.append_kv(k_pool, v_pool, summ, indptr, indices, np.array([0]),
                 np.array([0, 5]), toks, toks)
    if with_append:
        new = _np([ex["appended_key"]], np.float32)[:, None, :]
        qo.append_kv(k_pool, v_pool, summ, indptr, indices, np.array([5]),
                     np.array([0, 1]), new, new)
    return k_pool, summ, indptr, indices


def test_fig2_two_step(golden):
    ex = golden("fig2_two_step.json")
    pr = ex["printed"]
    _, summ, indptr, indices = _fig2_state(ex, with_append=False)
    q_t = _np(ex["q_t"], np.float32)[None, None, :]
    sc = qo.score_pages(q_t, summ, indptr, indices, group=1)
    assert sc[0].tolist() == [pr["U_A_qt"], pr["U_B_qt"]]
    sel, _, cnt = qo.select_topk(sc, indptr, indices, k=1)
    assert sel[0, 0, 0] == 0 and cnt[0, 0] == 1            # A
    q_t1 = _np(ex["q_t1"], np.float32)[None, None, :]
    assert qo.score_pages(q_t1, summ, indptr, indices, 1)[0, 1] == \
        pr["U_B_qt1_without_append"]

    _, summ, indptr, indices = _fig2_state(ex, with_append=True)
    assert summ[1, 0, 0].tolist() == pr["m_B_after"]
    assert summ[1, 0, 1].tolist() == pr["M_B_after"]
    sc = qo.score_pages(q_t1, summ, indptr, indices, group=1)
    assert sc[0].tolist() == [pr["U_A_qt1"], pr["U_B_qt1"]]
    sel, _, _ = qo.select_topk(sc, indptr, indices, k=1)
    assert sel[0, 0, 0] == 1                                # B


def test_four_page_selection(golden):
    ex = golden("four_page_selection.json")
    names = ex["pages"]
    for k, want in ex["selected"].items():
        got = qo.topk_pages(ex["U"], int(k))
        assert sorted(names[i] for i in got) == sorted(want)
    # eq (4) holds on every page of the example
    assert all(t <= u for t, u in zip(ex["true_max"], ex["U"]))


def test_byte_model(golden):
    ex = golden("byte_model.json")
    assert ex["budget_tokens"] // ex["S"] == ex["K"]
    assert qo.traffic_ratio(ex["L"], ex["S"], ex["K"]) == ex["rho"]
    dense, index, sel = qo.traffic_bytes(ex["vec_bytes"], ex["L"], ex["S"], ex["K"])
    mib = 1 << 20
    assert dense == ex["dense_MiB_per_layer_head"] * mib
    assert index == ex["index_MiB"] * mib
    assert sel == ex["selected_MiB"] * mib
    assert (index + sel) / dense == ex["rho"]


# --------------------------------------------------------------------------
# Summary: brute force, signed zero, tail lengths, slot reuse
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [np.float16, np.float32])
def test_summary_brute_force(dt):
    rng = np.random.default_rng(1)
    for n in (1, 2, 7, 16, 32):
        keys = rng.standard_normal((n, 64)).astype(dt)
        keys[keys == 0] = 1                                 # no signed-zero ambiguity
        m, M = qo.page_summary(keys)
        assert np.array_equal(m, keys.min(axis=0))
        assert np.array_equal(M, keys.max(axis=0))
        assert m.dtype == dt and M.dtype == dt


def test_summary_signed_zero_order():
    keys = np.array([[0.0, -0.0, -0.0], [-0.0, 0.0, -0.0]], np.float16)
    m, M = qo.page_summary(keys)
    assert np.signbit(m).tolist() == [True, True, True]
    assert np.signbit(M).tolist() == [False, False, True]


def _prefill(L, S, d=16, h=2, dt=np.float32, seed=0, poison=True):
    rng = np.random.default_rng(seed)
    P = -(-L // S)
    toks_k = rng.standard_normal((L, h, d)).astype(dt)
    toks_v = rng.standard_normal((L, h, d)).astype(dt)
    fill = np.nan if poison else 0
    k_pool = np.full((P + 2, h, S, d), fill, dt)
    v_pool = np.full((P + 2, h, S, d), fill, dt)
    summ = np.full((P + 2, h, 2, d), fill, dt)
    perm = rng.permutation(P + 2)[:P].astype(np.int32)
    indptr = np.array([0, P], np.int32)
    return toks_k, toks_v, k_pool, v_pool, summ, indptr, perm


@pytest.mark.parametrize("L", [1, 15, 16, 17, 33])
def test_append_tail_lengths(L):
    S = 16
    tk, tv, kp, vp, sm, indptr, perm = _prefill(L, S)
    qo.append_kv(kp, vp, sm, indptr, perm, np.array([0]), np.array([0, L]), tk, tv)
    P = -(-L // S)
    for p in range(P):
        valid = min(S, L - p * S)
        rows = tk[p * S:p * S + valid]                      # [valid, h, d]
        pp = perm[p]
        assert np.array_equal(sm[pp, :, 0], rows.min(axis=0))
        assert np.array_equal(sm[pp, :, 1], rows.max(axis=0))
        assert np.all(np.isfinite(sm[pp]))                  # poison never read
        assert np.array_equal(kp[pp, :, :valid], rows.transpose(1, 0, 2))
    # one token at a time (decode) reaches the same state as one prefill call
    tk2, tv2, kp2, vp2, sm2, _, _ = _prefill(L, S)
    for t in range(L):
        qo.append_kv(kp2, vp2, sm2, indptr, perm, np.array([t]), np.array([0, 1]),
                     tk[t:t + 1], tv[t:t + 1])
    for p in range(P):
        assert np.array_equal(sm2[perm[p]], sm[perm[p]])
    # build_summary over the pool is eq (1) over the same valid keys
    sm3 = qo.build_summary(kp, indptr, perm, np.array([L]))
    for p in range(P):
        assert np.array_equal(sm3[perm[p]], sm[perm[p]])


def test_slot_reuse_matches_fresh_page():
    """Allocate, fill, free, reallocate one physical slot (Quest page §3)."""
    S, d, h = 16, 8, 1
    rng = np.random.default_rng(3)
    old = (rng.standard_normal((S, h, d)) * 10).astype(np.float32)
    new = rng.standard_normal((5, h, d)).astype(np.float32)
    kp = np.zeros((1, h, S, d), np.float32)
    vp = np.zeros_like(kp)
    sm = np.zeros((1, h, 2, d), np.float32)
    ind = np.array([0, 1], np.int32)
    pages = np.array([0], np.int32)
    qo.append_kv(kp, vp, sm, ind, pages, np.array([0]), np.array([0, S]), old, old)
    qo.append_kv(kp, vp, sm, ind, pages, np.array([0]), np.array([0, 5]), new, new)
    fresh_k = np.zeros_like(kp)
    fresh_s = np.zeros_like(sm)
    qo.append_kv(fresh_k, np.zeros_like(kp), fresh_s, ind, pages, np.array([0]),
                 np.array([0, 5]), new, new)
    assert np.array_equal(sm, fresh_s)


# --------------------------------------------------------------------------
# Score: eq (4) invariant, closed forms, GQA reduction
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [np.float16, np.float32])
def test_bound_invariant_and_closed_forms(dt):
    rng = np.random.default_rng(7)
    for trial in range(200):
        d = int(rng.choice([2, 8, 64, 128]))
        n = int(rng.integers(1, 33))
        keys = (rng.standard_normal((n, d)) * rng.uniform(0.1, 8)).astype(dt)
        q = rng.standard_normal(d).astype(dt).astype(np.float64)
        m, M = qo.page_summary(keys)
        U = qo.page_bound(q, m, M)
        dots = keys.astype(np.float64) @ q
        tol = 1e-12 * (np.abs(q) @ np.maximum(np.abs(m), np.abs(M)).astype(np.float64))
        assert dots.max() <= U + tol                         # eq (4)
        # a one-key page is a point: the bound is that key's dot product
        U1 = qo.page_bound(q, *qo.page_summary(keys[:1]))
        assert abs(U1 - dots[0]) <= tol
        # q >= 0 picks M, q <= 0 picks m (text after eq (2))
        qp = np.abs(q)
        assert abs(qo.page_bound(qp, m, M) - qp @ M.astype(np.float64)) <= tol
        assert abs(qo.page_bound(-qp, m, M) - (-qp) @ m.astype(np.float64)) <= tol


def test_score_pages_group_reduction():
    rng = np.random.default_rng(11)
    h_kv, G, d, S = 2, 4, 16, 4
    summ = rng.standard_normal((6, h_kv, 2, d)).astype(np.float32)
    summ[:, :, 0], summ[:, :, 1] = (np.minimum(summ[:, :, 0], summ[:, :, 1]),
                                    np.maximum(summ[:, :, 0], summ[:, :, 1]))
    indptr = np.array([0, 2, 5], np.int32)
    indices = np.array([5, 0, 3, 1, 4], np.int32)
    q = rng.standard_normal((2, h_kv * G, d)).astype(np.float32)
    sc = qo.score_pages(q, summ, indptr, indices, group=G)
    # group == 1 per query head, then the group max, equals the grouped call
    per = [qo.score_pages(q[:, h:h + 1], summ[:, h // G:h // G + 1], indptr,
                          indices, 1)[0] for h in range(h_kv * G)]
    for g in range(h_kv):
        assert np.array_equal(sc[g], np.max(per[g * G:(g + 1) * G], axis=0))
    # direct eq (2)-(3) with explicit loops for one entry
    r, i, g = 1, 3, 1
    pp = indices[i]
    want = -np.inf
    for h in range(g * G, (g + 1) * G):
        tot = 0.0
        for j in range(d):
            a = float(q[r, h, j]) * float(summ[pp, g, 0, j])
            b = float(q[r, h, j]) * float(summ[pp, g, 1, j])
            tot += max(a, b)
        want = max(want, tot)
    assert abs(sc[g, i] - want) < 1e-12


def test_group_max_is_attained_by_brute_force():
    """Quest page §2.1 prints the shared score of a GQA group as
    U_{g,p} = max_{h in g} U_{h,p}. On pages built so that every head's bound
    is attained by a key of the page (its corner of the page's min/max box,
    eq (2)-(3)), the group score must equal the brute-force maximum over the
    group's heads and the page's valid keys of q_h . k in fp64: a
    characterisation that uses neither the bound's formula nor the group rule,
    and that a mean, a sum or a wrong head-to-group index breaks."""
    rng = np.random.default_rng(21)
    h_kv, G, d, S, P = 2, 4, 8, 16, 5
    L = P * S - 3                                       # a ragged tail page
    q = rng.standard_normal((1, h_kv * G, d)).astype(np.float32)
    perm = rng.permutation(P + 2)[:P].astype(np.int32)
    kp = np.full((P + 2, h_kv, S, d), np.nan, np.float32)
    for lp in range(P):
        n = min(S, L - lp * S)
        for g in range(h_kv):
            lo = rng.standard_normal(d).astype(np.float32)
            hi = (lo + rng.uniform(0.1, 2.0, d)).astype(np.float32)
            keys = [lo, hi] + [np.where(q[0, h] >= 0, hi, lo) for h in range(g * G, (g + 1) * G)]
            while len(keys) < n:                        # interior keys: the box is unchanged
                keys.append((lo + (hi - lo) * rng.uniform(0.05, 0.95, d)).astype(np.float32))
            kp[perm[lp], g, :n] = np.array(keys[:n])[rng.permutation(n)]
    indptr = np.array([0, P], np.int32)
    sm = qo.build_summary(kp, indptr, perm, np.array([L], np.int32))
    U = qo.score_pages(q, sm, indptr, perm, G)
    wrong_idx = wrong_mean = 0
    for lp in range(P):
        n = min(S, L - lp * S)
        for g in range(h_kv):
            keys = kp[perm[lp], g, :n].astype(np.float64)
            dots = keys @ q[0].astype(np.float64).T                 # [n, h_q]
            want = dots[:, g * G:(g + 1) * G].max()
            tol = 1e-12 * (np.abs(keys).max() * np.abs(q[0]).astype(np.float64).sum(axis=1).max())
            assert abs(U[g, lp] - want) <= tol
            # the rules a plausible mistake would compute differ here
            wrong_idx += abs(dots[:, g::h_kv].max() - want) > tol
            wrong_mean += abs(dots[:, g * G:(g + 1) * G].max(axis=0).mean() - want) > tol
    assert wrong_idx > 0 and wrong_mean > 0


# --------------------------------------------------------------------------
# Selection: brute-force rank characterisation, ties, K >= P
# --------------------------------------------------------------------------

def _rank_select(U, k):
    """Page i is chosen iff fewer than k pages beat it; a page beats i when its
    score is larger, or equal with a smaller index."""
    P = len(U)
    out = []
    for i in range(P):
        beats = sum(1 for j in range(P) if U[j] > U[i] or (U[j] == U[i] and j < i))
        if beats < k:
            out.append(i)
    return out


def test_select_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(400):
        P = int(rng.integers(1, 65))
        k = int(rng.integers(1, 70))
        if trial % 3 == 0:
            U = rng.integers(-3, 4, P).astype(np.float64)   # many ties
            U[U == 0] = rng.choice([0.0, -0.0], int((U == 0).sum()))
        else:
            U = rng.standard_normal(P)
        got = qo.topk_pages(U, k).tolist()
        assert got == _rank_select(U.tolist(), k)
        assert len(got) == min(k, P) and len(set(got)) == len(got)


def test_select_outputs_and_padding():
    U = np.array([[3.0, 1.0, 2.0, 2.0, -1.0]])
    indptr = np.array([0, 2, 5], np.int32)
    indices = np.array([9, 4, 7, 1, 0], np.int32)
    sl, sp, sc = qo.select_topk(U, indptr, indices, k=3)
    assert sl[0, 0].tolist() == [0, 1, -1] and sc[0, 0] == 2
    assert sp[0, 0].tolist() == [9, 4, -1]
    assert sl[1, 0].tolist() == [0, 1, 2] and sc[1, 0] == 3
    assert sp[1, 0].tolist() == [7, 1, 0]


# --------------------------------------------------------------------------
# Local window + sink + Quest hybrid budget (Quest page §2.2, §3.2)
# --------------------------------------------------------------------------

def test_hybrid_budget_split_of_the_page():
    # Quest page §2.2: a 2048-token budget keeps 512 recent tokens and 4
    # sinks, and spends the remaining 1532 tokens as whole pages on Quest.
    # At S = 16: 32 local pages, 1 sink page, floor(1532 / 16) = 95 pages.
    assert qo.hybrid_budget_pages(2048, 512, 4, 16) == (128, 32, 1, 95)
    assert 32 + 1 + 95 == 2048 // 16


def test_hybrid_brute_force():
    """Forced pages (first n_sink, last n_local of the P valid pages) are
    always chosen; every other chosen page beats every other unchosen page
    under (score desc, index asc); min(k, P) pages in ascending order."""
    rng = np.random.default_rng(11)
    for trial in range(600):
        P = int(rng.integers(1, 40))
        k = int(rng.integers(1, 45))
        n_sink = int(rng.integers(0, k + 1))
        n_local = int(rng.integers(0, k - n_sink + 1))
        U = (rng.integers(-3, 4, P).astype(np.float64) if trial % 3 == 0
             else rng.standard_normal(P))
        got = qo.hybrid_pages(U, P, k, n_sink, n_local).tolist()
        forced = {i for i in range(P) if i < n_sink or i >= P - n_local}
        assert got == sorted(set(got)) and len(got) == min(k, P)
        assert forced <= set(got)
        quest, out = set(got) - forced, set(range(P)) - set(got) - forced
        for c in quest:
            for x in out:
                assert (U[c], -c) > (U[x], -x)


def test_hybrid_reductions():
    rng = np.random.default_rng(12)
    for _ in range(100):
        P = int(rng.integers(1, 50))
        k = int(rng.integers(1, 60))
        U = rng.standard_normal(P)
        # nothing forced: plain Top-K (pinned by the rank characterisation)
        assert qo.hybrid_pages(U, P, k, 0, 0).tolist() == _rank_select(U.tolist(), k)
    # a short request: sink and window overlap and cover every page
    assert qo.hybrid_pages([0.1, 0.2, 0.3], 3, 8, 2, 2).tolist() == [0, 1, 2]
    # the window alone fills the budget: Quest gets nothing
    assert qo.hybrid_pages([9.0, 8.0, 7.0, 1.0, 0.5], 5, 2, 0, 2).tolist() == [3, 4]
    # one sink, one local, one Quest page (ties to the lower index)
    assert qo.hybrid_pages([1.0, 5.0, 5.0, 2.0], 4, 3, 1, 1).tolist() == [0, 1, 3]


def test_select_hybrid_outputs():
    U = np.array([[3.0, 1.0, 2.0, 2.0, -1.0, 0.5, 0.25]])
    indptr = np.array([0, 7], np.int32)
    indices = np.array([9, 4, 7, 1, 0, 3, 2], np.int32)
    # 6 valid pages (L = 90, S = 16): entry 6 is a reserved one and never competes
    sl, sp, sc = qo.select_hybrid(U, indptr, indices, np.array([90]), 16, k=4, n_sink=1, n_local=1)
    assert sl[0, 0].tolist() == [0, 2, 3, 5] and sc[0, 0] == 4
    assert sp[0, 0].tolist() == [9, 7, 1, 3]


# --------------------------------------------------------------------------
# Attention: library routine, K = P, eq (7), set semantics
# --------------------------------------------------------------------------

def test_dense_attention_matches_torch_sdpa():
    rng = np.random.default_rng(2)
    for L, d in ((1, 8), (37, 64), (300, 128)):
        q = rng.standard_normal(d)
        K = rng.standard_normal((L, d)) * 2
        V = rng.standard_normal((L, d))
        o, lse = qo.dense_attention(q, K, V)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q)[None, None, None], torch.tensor(K)[None, None],
            torch.tensor(V)[None, None])[0, 0, 0].numpy()
        assert np.allclose(o, ref, rtol=1e-12, atol=1e-13)
        s = K @ q / math.sqrt(d)
        assert abs(lse - np.log(np.exp(s).sum())) < 1e-10


def _paged_case(seed, lens, S=16, d=32, h_kv=2, G=1, dt=np.float16):
    rng = np.random.default_rng(seed)
    counts = [-(-L // S) for L in lens]
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    nnz = int(indptr[-1])
    perm = rng.permutation(nnz + 3)[:nnz].astype(np.int32)
    kp = np.full((nnz + 3, h_kv, S, d), np.nan, dt)
    vp = np.full_like(kp, np.nan)
    toks = []
    for r, L in enumerate(lens):
        k = rng.standard_normal((L, h_kv, d)).astype(dt)
        v = rng.standard_normal((L, h_kv, d)).astype(dt)
        for t in range(L):
            pp = perm[indptr[r] + t // S]
            kp[pp, :, t % S] = k[t]
            vp[pp, :, t % S] = v[t]
        toks.append((k, v))
    q = rng.standard_normal((len(lens), h_kv * G, d)).astype(dt)
    return kp, vp, indptr, perm, np.array(lens, np.int32), q, toks


def test_all_pages_equals_dense():
    lens = [1, 15, 16, 17, 100]
    kp, vp, indptr, perm, sl, q, toks = _paged_case(4, lens, G=2)
    G, h_kv = 2, 2
    sel = np.full((len(lens), h_kv, 8), -1, np.int32)
    for r, L in enumerate(lens):
        P = -(-L // 16)
        sel[r, :, :P] = np.arange(P)[::-1]                  # any order
    o, lse = qo.sparse_attention(q, kp, vp, indptr, perm, sl, sel, G)
    for r, (k, v) in enumerate(toks):
        for h in range(h_kv * G):
            od, ld = qo.dense_attention(q[r, h], k[:, h // G].astype(np.float64),
                                        v[:, h // G].astype(np.float64))
            assert np.allclose(o[r, h], od, rtol=1e-12, atol=1e-12)
            assert abs(lse[r, h] - ld) < 1e-10


def test_eq7_bound_and_set_semantics():
    rng = np.random.default_rng(9)
    lens = [200]
    kp, vp, indptr, perm, sl, q, toks = _paged_case(6, lens, d=64, h_kv=1)
    k, v = toks[0]
    P = 13
    for trial in range(30):
        chosen = np.sort(rng.choice(P, size=int(rng.integers(1, P)), replace=False))
        sel = np.full((1, 1, P), -1, np.int32)
        sel[0, 0, :len(chosen)] = rng.permutation(chosen)
        oc, _ = qo.sparse_attention(q, kp, vp, indptr, perm, sl, sel, 1)
        od, _ = qo.dense_attention(q[0, 0], k[:, 0], v[:, 0])
        mask = np.zeros(200, bool)
        for p in chosen:
            mask[p * 16:min(200, p * 16 + 16)] = True
        eps = qo.excluded_mass(q[0, 0], k[:, 0], mask, 1 / 8)
        vmax = qo.value_norm_max(v[:, 0])
        assert np.linalg.norm(od - oc[0, 0]) <= 2 * eps * vmax + 1e-9   # eq (7)
        # duplicates and -1 entries change nothing (set semantics)
        dup = np.concatenate([sel[0, 0], chosen[:1], [-1]])[None, None]
        od2, _ = qo.sparse_attention(q, kp, vp, indptr, perm, sl, dup, 1)
        assert np.array_equal(od2, oc)


def test_single_token_page_and_empty_set():
    kp, vp, indptr, perm, sl, q, toks = _paged_case(8, [17], d=16, h_kv=1)
    sel = np.array([[[1, -1]]], np.int32)                    # the 1-token tail page
    o, lse = qo.sparse_attention(q, kp, vp, indptr, perm, sl, sel, 1)
    assert np.array_equal(o[0, 0], toks[0][1][16, 0].astype(np.float64))
    sel = np.array([[[-1, -1]]], np.int32)
    o, lse = qo.sparse_attention(q, kp, vp, indptr, perm, sl, sel, 1)
    assert np.all(o == 0) and lse[0, 0] == -np.inf


def test_physical_shuffle_invariance():
    lens = [77]
    a = _paged_case(12, lens, d=16, h_kv=1)
    kp, vp, indptr, perm, sl, q, toks = a
    sel = np.array([[[0, 2, 4]]], np.int32)
    o1, _ = qo.sparse_attention(q, kp, vp, indptr, perm, sl, sel, 1)
    # move every page to a new physical slot
    newperm = perm[::-1].copy()
    kp2 = np.full_like(kp, np.nan)
    vp2 = np.full_like(vp, np.nan)
    kp2[newperm] = kp[perm]
    vp2[newperm] = vp[perm]
    o2, _ = qo.sparse_attention(q, kp2, vp2, indptr, newperm, sl, sel, 1)
    assert np.array_equal(o1, o2)


def test_combine_partials_is_global_softmax():
    rng = np.random.default_rng(13)
    q = rng.standard_normal(8)
    K = rng.standard_normal((40, 8)) * 3
    V = rng.standard_normal((40, 8))
    o, l = qo.dense_attention(q, K, V)
    cuts = [0, 5, 6, 23, 40]
    parts = [qo.dense_attention(q, K[a:b], V[a:b]) for a, b in zip(cuts, cuts[1:])]
    parts.append((np.zeros(8), -np.inf))                     # an empty piece
    oc, lc = qo.combine_partials(parts)
    assert np.allclose(oc, o, rtol=1e-12, atol=1e-13) and abs(lc - l) < 1e-12
    # a per-piece softmax then plain average is a different (wrong) answer
    avg = np.mean([p[0] for p in parts[:-1]], axis=0)
    assert np.abs(avg - o).max() > 1e-3


# --------------------------------------------------------------------------
# Planted mistakes: each plausible slip breaks at least one pin above
# --------------------------------------------------------------------------

def test_planted_mistakes_are_caught(golden, monkeypatch):
    ex = golden("worked_example_2d.json")
    keys = _np(ex["page"]["keys"], np.float32)
    q = _np(ex["q"])
    m, M = qo.page_summary(keys)
    slips = {
        "drop the max: q.M only": lambda q, m, M: float(np.dot(q, M)),
        "wrong sign on m": lambda q, m, M: float(np.maximum(-q * m, q * M).sum()),
        "min instead of max": lambda q, m, M: float(np.minimum(q * m, q * M).sum()),
        "swapped m/M per dim": lambda q, m, M: float(np.maximum(q * M[::-1], q * m[::-1]).sum()),
    }
    for name, f in slips.items():
        assert f(q, m, M) != ex["U"], name
    # a tie rule that prefers the higher index breaks the brute-force pin
    U = [1.0, 1.0, 0.5]
    wrong = sorted(np.lexsort((-np.arange(3), -np.asarray(U)))[:1].tolist())
    assert wrong != _rank_select(U, 1)


# ---------------------------------------------------------------------------
# Recall diagnostics (Quest page §1.1 recall paragraph and its four-page
# example; eq (6)-(7); §3.1 page slack)
# ---------------------------------------------------------------------------

def test_topr_tokens_brute_force():
    rng = np.random.default_rng(31)
    for trial in range(50):
        n = int(rng.integers(1, 40))
        s = rng.integers(-3, 4, size=n).astype(np.float64)          # many ties
        R = int(rng.integers(1, 50))
        want = sorted(range(n), key=lambda i: (-s[i], i))[:min(R, n)]
        assert list(qo.topr_tokens(s, R)) == want


def test_recall_four_page_example():
    """Pages A-D with true maxima 10, 3, 2, 1 and bounds 10, 14, 12, 4: K = 2
    takes B and C and misses the page of the highest logit; K = 3 recalls it."""
    logits = np.array([10., 0., 3., -1., 2., 0., 1., 0.])        # two tokens per page
    token_page = np.arange(8) // 2
    U = np.array([10., 14., 12., 4.])
    sel2 = qo.topk_pages(U, 2)
    assert sorted(sel2.tolist()) == [1, 2]
    assert qo.topr_page_recall(logits, token_page, sel2, 1) == 0.0
    assert qo.topr_page_recall(logits, token_page, sel2, 2) == 0.5   # 10 (A) and 3 (B)
    sel3 = qo.topk_pages(U, 3)
    assert sorted(sel3.tolist()) == [0, 1, 2]
    assert qo.topr_page_recall(logits, token_page, sel3, 1) == 1.0


def test_recall_diagnostics_special_cases():
    lens = [1, 16, 33, 70]
    kp, vp, indptr, perm, sl, q, toks = _paged_case(12, lens, G=2)
    G, h_kv, S = 2, 2, 16
    P = [-(-L // S) for L in lens]
    # every page selected: nothing excluded, every top token recalled
    full = np.full((len(lens), h_kv, 8), -1, np.int32)
    for r in range(len(lens)):
        full[r, :, :P[r]] = np.arange(P[r])
    d = qo.recall_diagnostics(q, kp, vp, indptr, perm, sl, full, G, R=5)
    assert np.all(d["eps"] == 0) and np.all(d["topr"] == 1)
    # a one-token page has an exact bound (m = M = k): slack 0 (request 0, and
    # the tail page of request 2); every slack is >= 0 (eq (4)); none past P
    assert np.all(d["slack"][:, indptr[0]] == 0)
    assert np.all(d["slack"][:, indptr[2] + 2] == 0)
    assert np.all(d["slack"] >= -1e-12)
    # V_max is the largest row norm of the request's values
    for r, (k, v) in enumerate(toks):
        for g in range(h_kv):
            assert d["vmax"][r, g] == np.linalg.norm(v[:, g].astype(np.float64), axis=-1).max()
    # nothing selected: all mass excluded, no top token recalled
    none = np.full((len(lens), h_kv, 8), -1, np.int32)
    d0 = qo.recall_diagnostics(q, kp, vp, indptr, perm, sl, none, G, R=3)
    assert np.allclose(d0["eps"], 1.0) and np.all(d0["topr"] == 0)
    # eq (7) on a partial selection: ||o - o_C|| <= 2 eps V_max
    part = full.copy()
    part[:, :, 1:] = -1                                              # first page only
    dp = qo.recall_diagnostics(q, kp, vp, indptr, perm, sl, part, G, R=3)
    oc, _ = qo.sparse_attention(q, kp, vp, indptr, perm, sl, part, G)
    for r, (k, v) in enumerate(toks):
        for h in range(h_kv * G):
            od, _ = qo.dense_attention(q[r, h], k[:, h // G], v[:, h // G])
            assert np.linalg.norm(od - oc[r, h]) <= 2 * dp["eps"][r, h] * dp["vmax"][r, h // G] + 1e-9


# ---------------------------------------------------------------------------
# FP8 (E4M3) summaries with directed rounding (Quest page §3, the paragraph on
# the summary dtype; §1.2 on keeping min/max in the quantized domain)
# ---------------------------------------------------------------------------

def test_e4m3_table_matches_torch_float8():
    """The oracle's decoding of all 256 codes equals torch's float8_e4m3fn
    (a library routine written independently of the oracle)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = qo.e4m3_values()
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_e4m3_closed_forms():
    v = qo.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0 and qo.E4M3_MAX == 448.0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0x30] == 0.5 and v[0xB8] == -1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert int((~np.isnan(v)).sum()) == 254


def _e4m3_test_values(seed):
    rng = np.random.default_rng(seed)
    ladder = np.unique(qo.e4m3_values()[~np.isnan(qo.e4m3_values())])
    x = np.concatenate([
        rng.standard_normal(4000) * 4.0,                   # the bulk
        rng.standard_normal(500) * 100.0,                  # large
        rng.standard_normal(500) * 2.0 ** -8,              # subnormal range
        ladder,                                            # every representable value
        (ladder[:-1] + ladder[1:]) / 2,                    # midpoints (RNE ties)
        [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -2.0 ** -10],
    ])
    x = np.clip(x, -448.0, 448.0).astype(np.float16).astype(np.float64)
    return x, ladder


def test_e4m3_directed_rounding_brackets_and_rne():
    x, ladder = _e4m3_test_values(7)
    d, od = qo.e4m3_round(x, -1)
    u, ou = qo.e4m3_round(x, +1)
    assert not od.any() and not ou.any()
    vd, vu = qo.e4m3_decode(d), qo.e4m3_decode(u)
    assert (vd <= x).all() and (vu >= x).all()
    # adjacent ladder values (or equal when x is representable)
    i = np.searchsorted(ladder, vd)
    exact = vd == vu
    assert np.array_equal(exact, np.isin(x, ladder))
    assert (ladder[np.minimum(i + 1, len(ladder) - 1)][~exact] == vu[~exact]).all()
    # torch's round-to-nearest-even lands on the nearer of the two
    rn = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert ((rn == vd) | (rn == vu)).all()
    lo, hi = x - vd, vu - x
    assert (rn[lo < hi] == vd[lo < hi]).all() and (rn[lo > hi] == vu[lo > hi]).all()
    # zero is stored as +0 whichever way it is rounded
    z = qo.e4m3_round(np.array([0.0, -0.0, 1e-6]), -1)[0]
    assert list(z) == [0, 0, 0]
    assert list(qo.e4m3_round(np.array([-0.0, -1e-6]), +1)[0]) == [0, 0]


def test_e4m3_overflow_flags_only_the_unbounded_side():
    c, o = qo.e4m3_round(np.array([449.0, 1e4, -449.0, -1e4]), -1)
    assert list(o) == [False, False, True, True]
    assert list(qo.e4m3_decode(c)) == [448.0, 448.0, -448.0, -448.0]
    c, o = qo.e4m3_round(np.array([449.0, -449.0]), +1)
    assert list(o) == [True, False]
    assert list(qo.e4m3_decode(c)) == [448.0, -448.0]


def test_e4m3_summary_keeps_the_bound():
    """The rounded-out box contains the page's keys, so U over it bounds the
    exact U and every q.k of the page (eq (4)), loosened by at most one
    E4M3 step per dimension (< |x| / 8 for |x| >= 2^-6, < 2^-9 below)."""
    rng = np.random.default_rng(11)
    d, S = 64, 16
    for trial in range(200):
        keys = rng.standard_normal((S, d)) * rng.choice([0.01, 1.0, 8.0])
        keys[:, :4] *= 8.0
        keys = keys.astype(np.float16)
        m, M = qo.page_summary(keys)
        summ = np.stack([m, M])
        codes, ovf = qo.summary_to_e4m3(summ)
        assert not ovf.any()
        m8, M8 = qo.e4m3_decode(codes[0]), qo.e4m3_decode(codes[1])
        assert (m8 <= m.astype(np.float64)).all() and (M8 >= M.astype(np.float64)).all()
        q = rng.standard_normal(d).astype(np.float16)
        U = qo.page_bound(q, m, M)
        U8 = qo.page_bound(q, m8, M8)
        true_max = (keys.astype(np.float64) @ q.astype(np.float64)).max()
        assert U8 >= U >= true_max - 1e-9
        mag = np.maximum(np.abs(m), np.abs(M)).astype(np.float64)
        step = np.where(mag >= 2.0 ** -6, mag / 8.0, 2.0 ** -9)
        assert U8 - U <= (np.abs(q.astype(np.float64)) * step).sum() + 1e-12


def test_e4m3_worked_example_is_on_the_grid(golden):
    """The 2-D example's box (-1,-2)..(3,4) is representable: U stays 8."""
    ex = golden("worked_example_2d.json")
    keys = _np(ex["page"]["keys"], np.float16)
    m, M = qo.page_summary(keys)
    codes, _ = qo.summary_to_e4m3(np.stack([m, M]))
    assert list(qo.e4m3_decode(codes[0])) == [-1.0, -2.0]
    assert list(qo.e4m3_decode(codes[1])) == [3.0, 4.0]
    q = _np(ex["q"])
    assert qo.page_bound(q, qo.e4m3_decode(codes[0]), qo.e4m3_decode(codes[1])) == 8.0


def test_e4m3_fold_in_code_domain_equals_rounded_exact_summary():
    """Keeping the FP8 summary up to date token by token in the code domain,
    m8 <- down(min(m8, k)) and M8 <- up(max(M8, k)), ends at the rounding of
    the exact summary: directed rounding is monotone, so it commutes with
    min/max. This is why an append may fold new keys straight into the codes."""
    rng = np.random.default_rng(5)
    d = 32
    for trial in range(50):
        n = int(rng.integers(1, 33))
        keys = (rng.standard_normal((n, d)) * 3).astype(np.float16)
        m8 = qo.e4m3_round(keys[0].astype(np.float64), -1)[0]
        M8 = qo.e4m3_round(keys[0].astype(np.float64), +1)[0]
        for t in range(1, n):
            k = keys[t].astype(np.float64)
            m8 = qo.e4m3_round(np.minimum(qo.e4m3_decode(m8), k), -1)[0]
            M8 = qo.e4m3_round(np.maximum(qo.e4m3_decode(M8), k), +1)[0]
        m, M = qo.page_summary(keys)
        codes, _ = qo.summary_to_e4m3(np.stack([m, M]))
        assert np.array_equal(m8, codes[0]) and np.array_equal(M8, codes[1])


def test_score_pages_e4m3_is_score_pages_of_the_decoded_box():
    kp, vp, indptr, perm, sl, q, toks = _paged_case(3, [40, 17], S=16, d=32, h_kv=2, G=2)
    summ = qo.build_summary(kp, indptr, perm, sl)
    codes, _ = qo.summary_to_e4m3(summ)
    a = qo.score_pages_e4m3(q, codes, indptr, perm, 2)
    b = qo.score_pages(q, summ, indptr, perm, 2)
    assert (a >= b - 1e-12).all()
    c = qo.score_pages(q, qo.e4m3_decode(codes), indptr, perm, 2)
    assert np.array_equal(a, c)


# ---------------------------------------------------------------------------
# GQA: per-query-head selection, per-KV-head union (Quest page §2.1, the MHA /
# GQA / head-sharing paragraphs)
# ---------------------------------------------------------------------------

def test_per_head_scores_bound_each_heads_dot_products():
    """U_{h,p} bounds every q_h.k of the page (eq (4) per head, brute force in
    fp64), and the group max of the per-head rows is the shared score."""
    lens = [70, 33]
    kp, vp, indptr, perm, sl, q, toks = _paged_case(12, lens, d=32, h_kv=2, G=4)
    sm = qo.build_summary(kp, indptr, perm, sl)
    U = qo.score_pages_per_head(q, sm, indptr, perm, 4)
    assert U.shape == (8, int(indptr[-1]))
    for r, (k, _) in enumerate(toks):
        for h in range(8):
            for lp in range(-(-lens[r] // 16)):
                keys = k[lp * 16:(lp + 1) * 16, h // 4].astype(np.float64)
                assert (keys @ q[r, h].astype(np.float64)).max() <= U[h, indptr[r] + lp] + 1e-12
    grp = qo.score_pages(q, sm, indptr, perm, 4)
    assert np.array_equal(U.reshape(2, 4, -1).max(axis=1), grp)
    # G = 1: the per-head rows are the MHA scores
    kp1, vp1, ip1, pm1, sl1, q1, _ = _paged_case(13, lens, d=32, h_kv=3, G=1)
    sm1 = qo.build_summary(kp1, ip1, pm1, sl1)
    assert np.array_equal(qo.score_pages_per_head(q1, sm1, ip1, pm1, 1),
                          qo.score_pages(q1, sm1, ip1, pm1, 1))


def test_union_pages_brute_force():
    rng = np.random.default_rng(21)
    for trial in range(200):
        G, K, P = int(rng.integers(1, 9)), int(rng.integers(1, 9)), int(rng.integers(1, 40))
        sel = np.full((G, K), -1, np.int64)
        for i in range(G):
            n = int(rng.integers(0, min(K, P) + 1))
            sel[i, :n] = rng.choice(P, size=n, replace=False)
        pages, masks = qo.union_pages(sel)
        want = sorted(set(int(x) for x in sel.ravel() if x >= 0))
        assert pages.tolist() == want and len(pages) <= G * K
        for p, m in zip(pages, masks):
            assert m == sum(1 << i for i in range(G) if p in sel[i])
    same = np.array([[4, 1, 7]] * 3)
    pages, masks = qo.union_pages(same)
    assert pages.tolist() == [1, 4, 7] and masks.tolist() == [7, 7, 7]


def test_per_head_attention_against_contiguous_tokens():
    """Each head's output is dense attention over the contiguous (un-paged)
    tokens of its own pages; with one set for the whole group it equals the
    shared-set attention."""
    rng = np.random.default_rng(23)
    lens = [90, 17]
    G, h_kv, K = 4, 2, 3
    kp, vp, indptr, perm, sl, q, toks = _paged_case(14, lens, d=32, h_kv=h_kv, G=G)
    sel = np.full((2, h_kv * G, K), -1, np.int32)
    for r, L in enumerate(lens):
        P = -(-L // 16)
        for h in range(h_kv * G):
            n = int(rng.integers(1, min(K, P) + 1))
            sel[r, h, :n] = rng.choice(P, size=n, replace=False)
    o, lse = qo.sparse_attention_per_head(q, kp, vp, indptr, perm, sl, sel, G)
    for r, (k, v) in enumerate(toks):
        for h in range(h_kv * G):
            rows = np.concatenate([np.arange(p * 16, min(lens[r], p * 16 + 16))
                                   for p in sorted(x for x in sel[r, h] if x >= 0)])
            od, ld = qo.dense_attention(q[r, h], k[rows, h // G].astype(np.float64),
                                        v[rows, h // G].astype(np.float64))
            assert np.allclose(o[r, h], od, rtol=1e-12, atol=1e-12)
            assert abs(lse[r, h] - ld) < 1e-10
    shared = sel[:, ::G]                                     # head 0's set for its group
    o2, _ = qo.sparse_attention_per_head(q, kp, vp, indptr, perm, sl, np.repeat(shared, G, axis=1), G)
    o3, _ = qo.sparse_attention(q, kp, vp, indptr, perm, sl, shared, G)
    assert np.array_equal(o2, o3)


def test_planted_mistakes_in_the_next_rows_are_caught(monkeypatch):
    """Plausible slips planted in the oracle's E4M3, per-head and union
    functions each make one of the pins above fail."""
    real_round, real_vals = qo.e4m3_round, qo.e4m3_values
    real_union, real_ph_attn = qo.union_pages, qo.sparse_attention_per_head

    def planted(attr, fake, pin, *args):
        monkeypatch.setattr(qo, attr, fake)
        with pytest.raises(AssertionError):
            pin(*args)
        monkeypatch.undo()

    # rounding toward the wrong side
    planted("e4m3_round", lambda x, toward: real_round(x, -toward),
            test_e4m3_directed_rounding_brackets_and_rne)

    # subnormals one binade off
    def vals_subnormal_slip():
        v = real_vals().copy()
        v[0x01:0x08] *= 2
        v[0x81:0x88] *= 2
        return v
    planted("e4m3_values", vals_subnormal_slip, test_e4m3_table_matches_torch_float8)

    # exponent bias 8 instead of 7
    def vals_bias_slip():
        v = real_vals().copy()
        v[0x08:0x7F] /= 2
        return v
    planted("e4m3_values", vals_bias_slip, test_e4m3_closed_forms)

    # head bits in the wrong order (a transposed index)
    planted("union_pages", lambda sel: real_union(np.asarray(sel)[::-1]),
            test_union_pages_brute_force)

    # every head of a group attending over the first head's pages
    def shared_set(q, kp, vp, ip, ix, sl, sel, group, sm_scale=None, requests=None):
        return real_ph_attn(q, kp, vp, ip, ix, sl, np.repeat(sel[:, ::group], group, axis=1),
                            group, sm_scale, requests)
    planted("sparse_attention_per_head", shared_set,
            test_per_head_attention_against_contiguous_tokens)

    # query head h read against KV head h % h_kv instead of h // group
    def wrong_kv_head(q, summary, indptr, indices, group, requests=None):
        h_kv = summary.shape[1]
        out = np.full((h_kv * group, int(indptr[-1])), np.nan)
        for r in range(len(indptr) - 1):
            lo, hi = int(indptr[r]), int(indptr[r + 1])
            phys = np.asarray(indices[lo:hi], dtype=np.int64)
            for h in range(h_kv * group):
                g = h % h_kv
                out[h, lo:hi] = qo.page_bound(q[r, h], summary[phys, g, 0], summary[phys, g, 1])
        return out
    planted("score_pages_per_head", wrong_kv_head,
            test_per_head_scores_bound_each_heads_dot_products)
