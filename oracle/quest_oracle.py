"""Plain, slow, fp64 CPU oracle for Quest-style query-aware page selection.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``query_aware_sparse_gb300``) never imports, calls or links
anything here, and nothing here imports the product path: the two share no
code, headers, tables or helpers.

Sources. "Quest page" is the PaperTrace chapter
"3.1.1 · Quest：用 min/max 上界筛选 KV 页"; "PageWeaver notes" is the reading
notes page "PageWeaver: KV-Guided Query Unions for Sparse Attention".
Each function names the section / equation it restates.

Conventions (where the pages are silent, the reading taken is stated here or
in the docstring of the function that takes it):

* Arrays are numpy. Keys/values/queries arrive in their stored dtype (float16
  or float32). Every floating-point *arithmetic* step runs in float64 on the
  exact fp64 image of the stored values. Min/max are selections, not
  arithmetic: the summary keeps the stored dtype and is exact.
* min/max use the total order of IEEE 754-2019 ``minimum``/``maximum`` on
  finite values, in which -0 < +0 (the pages are silent on signed zero).
* Layouts (one layer):
    k_pool, v_pool  [n_phys, h_kv, page_size, head_dim]
    summary         [n_phys, h_kv, 2, head_dim]   (index 0 = min m, 1 = max M)
    page_indptr     [batch + 1]   CSR row pointer into page_indices
    page_indices    [nnz]         physical page of logical page i of a request
    seq_lens        [batch]       valid tokens of each request
    q               [batch, h_kv * group, head_dim]
* ``score_pages`` with group > 1 takes the group max that Quest page §2.1
  prints, U_{g,p} = max_{h in g} U_{h,p} (one of the two aggregations the page
  weighs; the union is the other). Pinned by brute force on pages where each
  head's bound is attained by one of the page's keys.
"""

from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Signed-zero-aware min/max (the fold of Quest page §1.2 eq (8) / §3 eq (14))
# ---------------------------------------------------------------------------

def total_less(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise a < b in the order where -0 < +0 (finite inputs)."""
    a = np.asarray(a)
    b = np.asarray(b)
    return (a < b) | ((a == b) & np.signbit(a) & ~np.signbit(b))


def fold_min(cur: np.ndarray, k: np.ndarray) -> np.ndarray:
    """m <- min(m, k) of Quest page §1.2 eq (8), in the stored dtype."""
    return np.where(total_less(k, cur), k, cur).astype(cur.dtype)


def fold_max(cur: np.ndarray, k: np.ndarray) -> np.ndarray:
    """M <- max(M, k) of Quest page §1.2 eq (8), in the stored dtype."""
    return np.where(total_less(cur, k), k, cur).astype(cur.dtype)


def page_summary(keys: np.ndarray):
    """Per-dimension (m, M) of one page's valid keys, Quest page §1.1 eq (1).

    ``keys`` is [n_valid, head_dim] (n_valid >= 1). The box starts empty
    (min = +inf, max = -inf, Quest page §1.2) and folds each key in token order.
    """
    keys = np.asarray(keys)
    if keys.shape[0] < 1:
        raise ValueError("a page summary needs at least one valid key")
    m = np.full(keys.shape[1:], np.inf, dtype=keys.dtype)
    M = np.full(keys.shape[1:], -np.inf, dtype=keys.dtype)
    for r in range(keys.shape[0]):
        m = fold_min(m, keys[r])
        M = fold_max(M, keys[r])
    return m, M


# ---------------------------------------------------------------------------
# a1: cache append + incremental summary (Quest page §1.2 eq (8), §3 eq (14))
# ---------------------------------------------------------------------------

def append_kv(k_pool, v_pool, summary, page_indptr, page_indices,
              seq_lens_before, append_indptr, k_new, v_new):
    """Write new tokens into their pages and update the page summaries, in place.

    Token i of request r (append_indptr[r] <= i < append_indptr[r+1]) lands at
    position pos = seq_lens_before[r] + (i - append_indptr[r]), logical page
    pos // S, slot pos % S, physical page page_indices[page_indptr[r] + pos//S].
    Writing slot 0 opens the page: its summary restarts from the empty box
    (+inf min, -inf max), which is the same as m = M = k on the first write
    (Quest page §3) and makes a reused physical slot start fresh (Quest page
    §3, page recycling). Every other write folds the key in with eq (8).
    Slots that are never written are never read.
    """
    S = k_pool.shape[2]
    batch = len(seq_lens_before)
    for r in range(batch):
        for i in range(int(append_indptr[r]), int(append_indptr[r + 1])):
            pos = int(seq_lens_before[r]) + (i - int(append_indptr[r]))
            lp, slot = divmod(pos, S)
            if lp >= int(page_indptr[r + 1]) - int(page_indptr[r]):
                raise IndexError("append beyond the request's page table")
            pp = int(page_indices[int(page_indptr[r]) + lp])
            k_pool[pp, :, slot, :] = k_new[i]
            v_pool[pp, :, slot, :] = v_new[i]
            if slot == 0:
                summary[pp, :, 0, :] = np.inf
                summary[pp, :, 1, :] = -np.inf
            summary[pp, :, 0, :] = fold_min(summary[pp, :, 0, :], k_new[i])
            summary[pp, :, 1, :] = fold_max(summary[pp, :, 1, :], k_new[i])


def build_summary(k_pool, page_indptr, page_indices, seq_lens, summary=None,
                  requests=None):
    """Summaries of every page of the listed requests from the pool's valid keys.

    Eq (1) of Quest page §1.1 over each page's valid tokens only (the tail page
    holds min(S, L - p*S) of them, Quest page §1.2). Vectorised over pages and
    heads; the fold over slots is the same eq (8) fold as ``append_kv``.
    """
    n_phys, h_kv, S, d = k_pool.shape
    if summary is None:
        summary = np.zeros((n_phys, h_kv, 2, d), dtype=k_pool.dtype)
    reqs = range(len(seq_lens)) if requests is None else requests
    for r in reqs:
        lo, hi = int(page_indptr[r]), int(page_indptr[r + 1])
        L = int(seq_lens[r])
        n_pages = -(-L // S)
        if n_pages > hi - lo:
            raise ValueError("seq_len exceeds the request's page table")
        if n_pages == 0:
            continue
        phys = np.asarray(page_indices[lo:lo + n_pages], dtype=np.int64)
        valid = np.minimum(S, L - np.arange(n_pages) * S)          # [n_pages]
        m = np.full((n_pages, h_kv, d), np.inf, dtype=k_pool.dtype)
        M = np.full((n_pages, h_kv, d), -np.inf, dtype=k_pool.dtype)
        for slot in range(S):
            live = valid > slot
            if not live.any():
                break
            k = k_pool[phys[live], :, slot, :]
            m[live] = fold_min(m[live], k)
            M[live] = fold_max(M[live], k)
        summary[phys, :, 0, :] = m
        summary[phys, :, 1, :] = M
    return summary


# ---------------------------------------------------------------------------
# a2: page upper bound U_p(q) (Quest page §1.1 eq (2)-(3)); GQA group max (§2.1)
# ---------------------------------------------------------------------------

def page_bound(q, m, M):
    """U_p(q) = sum_j max(q_j m_j, q_j M_j) in fp64 (Quest page §1.1 eq (2)-(3)).

    q is [d]; m, M are [..., d]. Returns [...].
    """
    q = np.asarray(q, dtype=F64)
    m = np.asarray(m, dtype=F64)
    M = np.asarray(M, dtype=F64)
    return np.maximum(q * m, q * M).sum(axis=-1)


def score_pages(q, summary, page_indptr, page_indices, group, requests=None,
                heads=None):
    """Scores [h_kv, nnz] (fp64) for every page of every request.

    For KV head g the score of a page is U of that page under each query head
    h in g*group .. g*group+group-1; with group > 1 the group shares one page
    set and its score is max_h U_{h,p} (Quest page §2.1, the group max the
    GQA discussion prints). Pages outside the
    listed requests / heads are left NaN.
    """
    n_phys, h_kv, _, d = summary.shape
    batch = len(page_indptr) - 1
    nnz = int(page_indptr[batch])
    scores = np.full((h_kv, nnz), np.nan, dtype=F64)
    reqs = range(batch) if requests is None else requests
    hs = range(h_kv) if heads is None else heads
    for r in reqs:
        lo, hi = int(page_indptr[r]), int(page_indptr[r + 1])
        if hi == lo:
            continue
        phys = np.asarray(page_indices[lo:hi], dtype=np.int64)
        for g in hs:
            m = summary[phys, g, 0, :]
            M = summary[phys, g, 1, :]
            best = np.full(hi - lo, -np.inf)
            for h in range(g * group, (g + 1) * group):
                best = np.maximum(best, page_bound(q[r, h], m, M))
            scores[g, lo:hi] = best
    return scores


# ---------------------------------------------------------------------------
# a3: fixed-budget Top-K pages (Quest page Fig. 1, §1.1 four-page example)
# ---------------------------------------------------------------------------

def topk_pages(U, k):
    """Logical indices of the K largest scores, ties to the lower index.

    Sort by (score descending, index ascending) and keep the first min(K, P);
    the chosen indices are returned in ascending order. -0 and +0 compare
    equal, so the index decides between them.
    """
    U = np.asarray(U, dtype=F64)
    P = U.shape[0]
    order = np.lexsort((np.arange(P), -U))
    return np.sort(order[:min(k, P)])


def select_topk(scores, page_indptr, page_indices, k, requests=None):
    """Per (request, KV head): Top-K logical pages, their physical pages, count.

    Returns sel_logical, sel_phys [batch, h_kv, k] (int32, -1 padded) and
    sel_count [batch, h_kv] = min(k, P_r).
    """
    h_kv = scores.shape[0]
    batch = len(page_indptr) - 1
    sel_logical = np.full((batch, h_kv, k), -1, dtype=np.int32)
    sel_phys = np.full((batch, h_kv, k), -1, dtype=np.int32)
    sel_count = np.zeros((batch, h_kv), dtype=np.int32)
    reqs = range(batch) if requests is None else requests
    for r in reqs:
        lo, hi = int(page_indptr[r]), int(page_indptr[r + 1])
        for g in range(h_kv):
            chosen = topk_pages(scores[g, lo:hi], k)
            n = len(chosen)
            sel_logical[r, g, :n] = chosen
            sel_phys[r, g, :n] = np.asarray(page_indices, dtype=np.int64)[lo + chosen]
            sel_count[r, g] = n
    return sel_logical, sel_phys, sel_count


def forced_pages(P, n_sink, n_local):
    """Pages kept whatever their score: the first n_sink (sink) and the last
    n_local (local window, tail page included) of the P valid pages, as one
    set (Quest page §3.2: C_local and C_sink may overlap; pages are counted
    after the union)."""
    return sorted(set(range(min(n_sink, P))) | set(range(max(0, P - n_local), P)))


def hybrid_pages(U, P, k, n_sink, n_local):
    """C = C_local ∪ C_sink ∪ C_quest (Quest page §3.2; budget split of §2.2).

    The forced pages are always chosen; the remaining budget k - |forced|
    goes to Quest: the other valid pages (index < P) ranked by (score
    descending, index ascending). The chosen indices are returned in
    ascending order; there are min(k, P) of them. Requires
    n_sink + n_local <= k.
    """
    U = np.asarray(U, dtype=F64)
    forced = forced_pages(P, n_sink, n_local)
    assert len(forced) <= k
    rest = np.array([i for i in range(P) if i not in set(forced)], dtype=np.int64)
    order = rest[np.lexsort((rest, -U[rest]))] if len(rest) else rest
    quest = order[:max(0, min(k, P) - len(forced))]
    return np.sort(np.concatenate([np.asarray(forced, dtype=np.int64), quest]))


def select_hybrid(scores, page_indptr, page_indices, seq_lens, page_size, k, n_sink, n_local,
                  requests=None):
    """select_topk with the local window + sink pages forced (hybrid_pages);
    only the P_r = ceil(L_r / S) valid pages of each request compete.
    n_sink = n_local = 0 is plain Quest Top-K over the valid pages."""
    h_kv = scores.shape[0]
    batch = len(page_indptr) - 1
    sel_logical = np.full((batch, h_kv, k), -1, dtype=np.int32)
    sel_phys = np.full((batch, h_kv, k), -1, dtype=np.int32)
    sel_count = np.zeros((batch, h_kv), dtype=np.int32)
    reqs = range(batch) if requests is None else requests
    for r in reqs:
        lo = int(page_indptr[r])
        P = min(-(-int(seq_lens[r]) // page_size), int(page_indptr[r + 1]) - lo)
        for g in range(h_kv):
            chosen = hybrid_pages(scores[g, lo:lo + P], P, k, n_sink, n_local)
            n = len(chosen)
            sel_logical[r, g, :n] = chosen
            sel_phys[r, g, :n] = np.asarray(page_indices, dtype=np.int64)[lo + chosen]
            sel_count[r, g] = n
    return sel_logical, sel_phys, sel_count


def hybrid_budget_pages(budget_tokens, local_tokens, sink_tokens, page_size):
    """Page counts of the budget split in Quest page §2.2: local window and
    sinks in whole pages (ceil), the rest of the token budget as whole pages
    for Quest (floor). Returns (k, n_local, n_sink, quest_pages)."""
    n_local = -(-local_tokens // page_size)
    n_sink = -(-sink_tokens // page_size)
    quest = (budget_tokens - local_tokens - sink_tokens) // page_size
    return n_local + n_sink + quest, n_local, n_sink, quest


# ---------------------------------------------------------------------------
# a4/a5: attention over a candidate page set (Quest page Fig. 1, eq (6);
#        PageWeaver notes §2 eq (1)-(2) for the exact token set and 1/sqrt(d))
# ---------------------------------------------------------------------------

def softmax_attention(q, keys, values, sm_scale):
    """o = sum_t softmax(q.k_t * scale) v_t and lse over the given rows (fp64).

    An empty key set gives o = 0 and lse = -inf (PageWeaver notes §2).
    """
    q = np.asarray(q, dtype=F64)
    keys = np.asarray(keys, dtype=F64)
    values = np.asarray(values, dtype=F64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1]), -np.inf
    s = (keys @ q) * sm_scale
    mx = s.max()
    p = np.exp(s - mx)
    z = p.sum()
    return (p @ values) / z, mx + math.log(z)


def candidate_tokens(k_pool, v_pool, page_indptr, page_indices, seq_lens, r, g,
                     logical_pages):
    """Keys/values of the valid tokens of the given logical pages of request r.

    The list is a set: -1 entries are skipped and repeats add nothing
    (PageWeaver notes §2). The tail page contributes only its valid tokens
    (Quest page §1.2, last_page_len).
    """
    S = k_pool.shape[2]
    L = int(seq_lens[r])
    lo = int(page_indptr[r])
    lps = sorted({int(x) for x in logical_pages if int(x) >= 0})
    ks, vs = [], []
    for lp in lps:
        valid = min(S, L - lp * S)
        if valid <= 0:
            raise IndexError("selected page holds no valid token")
        pp = int(page_indices[lo + lp])
        ks.append(k_pool[pp, g, :valid, :])
        vs.append(v_pool[pp, g, :valid, :])
    d = k_pool.shape[3]
    if not ks:
        return np.zeros((0, d)), np.zeros((0, d))
    return np.concatenate(ks).astype(F64), np.concatenate(vs).astype(F64)


def sparse_attention(q, k_pool, v_pool, page_indptr, page_indices, seq_lens,
                     sel_logical, group, sm_scale=None, requests=None):
    """o [batch, h_q, d] and lse [batch, h_q] over each head's candidate set.

    Query head h uses the set chosen for its KV head h // group; the softmax
    denominator covers only the valid candidate tokens, so the result is the
    renormalised approximation of eq (6) (Quest page Fig. 1, §1.1).
    Rows of requests not listed are NaN.
    """
    batch, h_q, d = q.shape
    h_kv = k_pool.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    o = np.full((batch, h_q, d), np.nan)
    lse = np.full((batch, h_q), np.nan)
    reqs = range(batch) if requests is None else requests
    for r in reqs:
        for g in range(h_kv):
            keys, vals = candidate_tokens(k_pool, v_pool, page_indptr,
                                          page_indices, seq_lens, r, g,
                                          sel_logical[r, g])
            for h in range(g * group, (g + 1) * group):
                o[r, h], lse[r, h] = softmax_attention(q[r, h], keys, vals,
                                                       sm_scale)
    return o, lse


def dense_attention(q, keys, values, sm_scale=None):
    """Plain attention of one query over contiguous, un-paged K/V (fp64)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(np.asarray(q).shape[-1])
    return softmax_attention(q, keys, values, sm_scale)


def combine_partials(partials):
    """Merge (o_c, lse_c) pieces of one row by log-sum-exp (Quest page §2.1).

    Each piece is the attention over a disjoint token subset; the merge uses
    the row's global maximum, never a per-piece softmax average.
    """
    live = [(o, l) for o, l in partials if l != -np.inf]
    if not live:
        d = len(partials[0][0]) if partials else 0
        return np.zeros(d), -np.inf
    mx = max(l for _, l in live)
    w = np.array([math.exp(l - mx) for _, l in live])
    o = sum(wi * np.asarray(oi, dtype=F64) for wi, (oi, _) in zip(w, live))
    return o / w.sum(), mx + math.log(w.sum())


# ---------------------------------------------------------------------------
# Diagnostics (Quest page §1.1 eq (6)-(7), §3.1 page slack)
# ---------------------------------------------------------------------------

def excluded_mass(q, keys, mask, sm_scale):
    """epsilon = dense softmax mass of the tokens outside the candidate set."""
    s = (np.asarray(keys, dtype=F64) @ np.asarray(q, dtype=F64)) * sm_scale
    p = np.exp(s - s.max())
    p /= p.sum()
    return float(p[~np.asarray(mask, dtype=bool)].sum())


def value_norm_max(values):
    """V_max = max_t ||v_t||_2 (Quest page §1.1, eq (7))."""
    return float(np.linalg.norm(np.asarray(values, dtype=F64), axis=-1).max())


def page_slack(q, keys):
    """g_p(q) = U_p(q) - max_r q.k_r >= 0 for one page (Quest page §3.1)."""
    keys = np.asarray(keys)
    m, M = page_summary(keys)
    return float(page_bound(q, m, M) - (keys.astype(F64) @ np.asarray(q, F64)).max())


def topr_tokens(logits, R):
    """Indices of the min(R, n) largest logits, ties to the lower index (the
    select's order rule, applied to tokens)."""
    s = np.asarray(logits, dtype=F64)
    order = np.lexsort((np.arange(len(s)), -s))
    return order[:min(R, len(s))]


def topr_page_recall(logits, token_page, selected_pages, R):
    """Top-R token recall (Quest page §1.1, recall paragraph): the share of the
    R tokens with the highest dense logits whose page is a selected page."""
    top = topr_tokens(logits, R)
    sel = {int(p) for p in selected_pages if int(p) >= 0}
    return sum(int(token_page[i]) in sel for i in top) / len(top)


def recall_diagnostics(q, k_pool, v_pool, page_indptr, page_indices, seq_lens,
                       sel_logical, group, R, sm_scale=None):
    """Per-query-head diagnostics of a selection against dense attention over
    each request's valid tokens (Quest page §1.1 eq (6)-(7) and its recall
    paragraph; §3.1 page slack). Query head h uses the pages chosen for its
    KV head h // group.

    slack [h_q, nnz]    g_p(q_h) = U_p(q_h) - max over the page's valid keys
                        of q_h.k (unscaled); NaN past a request's pages
    eps   [batch, h_q]  dense softmax mass outside the candidate pages
    topr  [batch, h_q]  top-R token recall of the candidate pages
    vmax  [batch, h_kv] max_t ||v_t||_2
    """
    batch, h_q, d = q.shape
    h_kv, S = k_pool.shape[1], k_pool.shape[2]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    slack = np.full((h_q, len(page_indices)), np.nan)
    eps = np.full((batch, h_q), np.nan)
    topr = np.full((batch, h_q), np.nan)
    vmax = np.full((batch, h_kv), np.nan)
    for r in range(batch):
        L = int(seq_lens[r])
        P = -(-L // S)
        lo = int(page_indptr[r])
        token_page = np.arange(L) // S
        for g in range(h_kv):
            keys, vals = candidate_tokens(k_pool, v_pool, page_indptr, page_indices,
                                          seq_lens, r, g, range(P))
            sel = [int(p) for p in sel_logical[r, g] if int(p) >= 0]
            mask = np.isin(token_page, sel)
            vmax[r, g] = value_norm_max(vals)
            for h in range(g * group, (g + 1) * group):
                qh = q[r, h]
                eps[r, h] = excluded_mass(qh, keys, mask, sm_scale)
                topr[r, h] = topr_page_recall(keys @ np.asarray(qh, dtype=F64),
                                              token_page, sel, R)
                for lp in range(P):
                    pp = int(page_indices[lo + lp])
                    slack[h, lo + lp] = page_slack(qh, k_pool[pp, g, :min(S, L - lp * S)])
    return dict(slack=slack, eps=eps, topr=topr, vmax=vmax)


# ---------------------------------------------------------------------------
# GQA with per-query-head selection and a per-KV-head union (Quest page §2.1,
# the MHA / GQA / head-sharing paragraphs: each query head picks its own
# pages, the shared KV head reads the union of the picks once, and each head's
# attention still runs over its own set only)
# ---------------------------------------------------------------------------

def score_pages_per_head(q, summary, page_indptr, page_indices, group, requests=None):
    """Scores [h_q, nnz] (fp64): U_{h,p} of every query head h against the
    summary of its KV head h // group, with no aggregation over the group."""
    n_phys, h_kv, _, d = summary.shape
    batch = len(page_indptr) - 1
    nnz = int(page_indptr[batch])
    scores = np.full((h_kv * group, nnz), np.nan, dtype=F64)
    reqs = range(batch) if requests is None else requests
    for r in reqs:
        lo, hi = int(page_indptr[r]), int(page_indptr[r + 1])
        if hi == lo:
            continue
        phys = np.asarray(page_indices[lo:hi], dtype=np.int64)
        for h in range(h_kv * group):
            g = h // group
            scores[h, lo:hi] = page_bound(q[r, h], summary[phys, g, 0, :], summary[phys, g, 1, :])
    return scores


def union_pages(sel_heads):
    """Union of the page sets of one KV head's query heads.

    sel_heads: [G, K] logical ids (-1 = empty slot). Returns (pages, masks):
    the distinct ids in increasing order and, per page, the bit set of the
    heads (bit i = head i of the group) that chose it.
    """
    owners = {}
    for i, row in enumerate(np.asarray(sel_heads)):
        for lp in row:
            lp = int(lp)
            if lp >= 0:
                owners[lp] = owners.get(lp, 0) | (1 << i)
    pages = sorted(owners)
    return np.array(pages, dtype=np.int64), np.array([owners[p] for p in pages], dtype=np.int64)


def sparse_attention_per_head(q, k_pool, v_pool, page_indptr, page_indices, seq_lens,
                              sel_logical, group, sm_scale=None, requests=None):
    """o [batch, h_q, d] and lse [batch, h_q] with a page set per query head.

    sel_logical is [batch, h_q, K]: query head h attends over the valid tokens
    of its own pages, read from its KV head h // group (the union only decides
    which pages are fetched, never which tokens a head weighs).
    """
    batch, h_q, d = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    o = np.full((batch, h_q, d), np.nan)
    lse = np.full((batch, h_q), np.nan)
    reqs = range(batch) if requests is None else requests
    for r in reqs:
        for h in range(h_q):
            keys, vals = candidate_tokens(k_pool, v_pool, page_indptr, page_indices, seq_lens,
                                          r, h // group, sel_logical[r, h])
            o[r, h], lse[r, h] = softmax_attention(q[r, h], keys, vals, sm_scale)
    return o, lse


# ---------------------------------------------------------------------------
# FP8 (E4M3) page summaries with directed rounding (Quest page §3, the
# paragraph on the summary dtype: min rounded toward -inf, max toward +inf,
# so the stored box still contains the page's keys and eq (4) stays a bound)
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_values():
    """The real value of each of the 256 E4M3 codes (NaN for the NaN codes).

    Format (OCP 8-bit floating point, E4M3 variant without infinities): bit 7
    sign, bits 6..3 exponent field e (bias 7), bits 2..0 mantissa m. e = 0 is
    subnormal, (m / 8) * 2^-6; otherwise (1 + m / 8) * 2^(e - 7); e = 15 with
    m = 7 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    out = np.empty(256, dtype=F64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 15 and m == 7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def _e4m3_ladder():
    """Finite E4M3 values in increasing order with their codes; zero appears
    once, as code 0x00 (reading: a rounded zero is stored as +0)."""
    vals = e4m3_values()
    codes = [c for c in range(256) if not np.isnan(vals[c]) and c != 0x80]
    codes.sort(key=lambda c: vals[c])
    return vals[codes], np.array(codes, dtype=np.uint8)


def e4m3_round(x, toward):
    """Directed rounding of finite reals into E4M3 codes.

    toward = -1: the largest E4M3 value <= x; toward = +1: the smallest
    E4M3 value >= x. Exactly representable x keep their value. Returns
    (codes uint8, overflow bool): where no E4M3 value lies on the required
    side (x < -448 rounding down, x > 448 rounding up) the code saturates at
    -448 / +448 and overflow is set, since the result then no longer bounds x.
    """
    x = np.asarray(x, dtype=F64)
    ladder, codes = _e4m3_ladder()
    if toward < 0:
        i = np.searchsorted(ladder, x, side="right") - 1
        ovf = i < 0
    else:
        i = np.searchsorted(ladder, x, side="left")
        ovf = i >= len(ladder)
    i = np.clip(i, 0, len(ladder) - 1)
    return codes[i], ovf


def e4m3_decode(codes):
    """fp64 value of E4M3 codes."""
    return e4m3_values()[np.asarray(codes, dtype=np.int64)]


def summary_to_e4m3(summary):
    """FP8 summary of an exact one: [..., 0, :] (min) rounded toward -inf,
    [..., 1, :] (max) toward +inf. Returns (codes uint8 of the same shape,
    overflow bool of the same shape)."""
    summary = np.asarray(summary)
    codes = np.empty(summary.shape, dtype=np.uint8)
    ovf = np.zeros(summary.shape, dtype=bool)
    codes[..., 0, :], ovf[..., 0, :] = e4m3_round(summary[..., 0, :], -1)
    codes[..., 1, :], ovf[..., 1, :] = e4m3_round(summary[..., 1, :], +1)
    return codes, ovf


def score_pages_e4m3(q, summary_codes, page_indptr, page_indices, group, requests=None,
                     heads=None):
    """score_pages over the decoded FP8 summary: U of the rounded-out box."""
    return score_pages(q, e4m3_decode(summary_codes), page_indptr, page_indices, group,
                       requests=requests, heads=heads)


# ---------------------------------------------------------------------------
# Byte model (Quest page §2 eq (9)-(12))
# ---------------------------------------------------------------------------

def traffic_ratio(L, S, K):
    """rho = (T_index + T_selected) / T_dense = 1/S + K S / L (eq (12))."""
    return 1.0 / S + K * S / L


def traffic_bytes(vec_bytes, L, S, K):
    """(T_dense, T_index, T_selected) in bytes, eq (9)-(11); M = vec_bytes."""
    P = L / S
    return 2 * vec_bytes * L, 2 * vec_bytes * P, 2 * vec_bytes * K * S
