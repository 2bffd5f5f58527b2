"""Full-size workloads through the CUDA path, checked against the oracle.

Each test builds the workload's cache through the library (prefill with
quest_append_kv), runs decode steps with quest_decode_step (the launch the
bench times) and, where noted, the unfused four calls, then recomputes
(request, KV head) units with the oracle from the generated tokens: summaries
bit-exact, scores within the score tolerance, selections under the near-tie
rule, attention within 2e-3 of fp64 (every head of the 32K layer and of three
of the sixteen GQA requests; two heads of the 128K steps). Every unit's
selection is also checked exactly against the oracle's Top-K over the GPU's
own fp32 scores.
"""

import math

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quest_oracle as qo
from tests._cases import attn_close, dev_i32, np_of

pytestmark = pytest.mark.gpu


def _gpu_cache(table, w):
    import query_aware_sparse_gb300 as qs
    kp, vp, sm = wl.empty_pool(table, w.h_kv, w.head_dim, w.dtype, device="cuda", poison=False)
    return qs.PagedCache(kp, vp, sm)


def _table(table, seq_lens):
    import query_aware_sparse_gb300 as qs
    return qs.PageTable(dev_i32(table.page_indptr), dev_i32(table.page_indices),
                        dev_i32(np.asarray(seq_lens, np.int32)), nnz=table.nnz)


class Unit:
    """Oracle view of one request restricted to a few KV heads."""

    def __init__(self, k_tok, v_tok, q_rows, heads, group, S):
        self.heads, self.G, self.S = list(heads), group, S
        self.k = np_of(k_tok)                  # [L, nh, d] stored values
        self.v = np_of(v_tok)
        self.q = np_of(q_rows)                 # [nh * G, d]

    def oracle(self, L, K):
        S, nh, d = self.S, len(self.heads), self.k.shape[-1]
        t = wl.make_page_table([L], S)
        kp, vp, _ = wl.empty_pool(t, nh, d, torch.from_numpy(self.k).dtype, poison=True)
        ind = np.array([0, L])
        wl.place_tokens(kp, t, torch.from_numpy(self.k[:L]), ind)
        wl.place_tokens(vp, t, torch.from_numpy(self.v[:L]), ind)
        kp, vp = kp.numpy(), vp.numpy()
        sm = qo.build_summary(kp, t.page_indptr, t.page_indices, np.array([L]))
        sc = qo.score_pages(self.q[None], sm, t.page_indptr, t.page_indices, self.G)
        sel, _, _ = qo.select_topk(sc, t.page_indptr, t.page_indices, K)
        return dict(t=t, kp=kp, vp=vp, sm=sm, sc=sc, sel=sel)

    def check(self, ref, L, K, g_summary, g_scores, g_sel, g_cnt, g_out, g_lse, phys):
        """Compare GPU rows (already sliced to this request and these heads)."""
        S = self.S
        P = -(-L // S)
        # summaries: bit-exact on every page of the sampled heads
        gs = g_summary[phys[:P]][:, self.heads]          # [P, nh, 2, d]
        assert np.array_equal(gs.view(np.uint16 if gs.dtype == np.float16 else np.uint32),
                              ref["sm"][:P].view(np.uint16 if gs.dtype == np.float16 else np.uint32))
        # scores
        mag = np.maximum(np.abs(ref["sm"][:P, :, 0].astype(np.float64)),
                         np.abs(ref["sm"][:P, :, 1].astype(np.float64)))
        qa = np.abs(self.q.astype(np.float64))
        for j, h in enumerate(self.heads):
            tol = 1e-4 * np.max([mag[:, j] @ qa[j * self.G + x] for x in range(self.G)], axis=0)
            assert np.all(np.abs(g_scores[j, :P] - ref["sc"][j, :P]) <= tol), (h, np.max(np.abs(g_scores[j, :P] - ref["sc"][j, :P]) / tol))
            # selection: identical sets except near-ties of the K-th score
            want = set(qo.topk_pages(ref["sc"][j, :P], K).tolist())
            got_l = [int(x) for x in g_sel[j] if x >= 0]
            got = set(got_l)
            assert len(got) == len(got_l) == min(K, P) == int(g_cnt[j])
            if P > K:
                kth = np.sort(ref["sc"][j, :P])[::-1][K - 1]
                for p in got ^ want:
                    assert abs(ref["sc"][j, p] - kth) <= tol[p] + 1e-9, (h, p)
        # attention on the GPU's (now validated) sets
        sel = np.full((1, len(self.heads), max(K, 1)), -1, np.int32)
        for j in range(len(self.heads)):
            ids = [int(x) for x in g_sel[j] if x >= 0]
            sel[0, j, :len(ids)] = ids
        ro, rl = qo.sparse_attention(self.q[None], ref["kp"], ref["vp"], ref["t"].page_indptr,
                                     ref["t"].page_indices, np.array([L]), sel, self.G)
        ok, rel = attn_close(g_out, ro[0])
        assert ok.all(), rel.max()
        assert np.allclose(g_lse, rl[0], rtol=1e-4, atol=1e-4)


def check_every_selection(scores, sel_logical, sel_count, table, seq_lens, K):
    """Every (request, KV head) selection equals the oracle's Top-K taken over
    the GPU's own fp32 scores (the same precision on both sides, so the sets
    must agree exactly, ties to the lower page)."""
    S = table.page_size
    for r in range(len(seq_lens)):
        lo = int(table.page_indptr[r])
        P = -(-int(seq_lens[r]) // S)
        for g in range(scores.shape[0]):
            want = qo.topk_pages(scores[g, lo:lo + P].astype(np.float64), K)
            got = [int(x) for x in sel_logical[r, g] if x >= 0]
            assert int(sel_count[r, g]) == len(got) == min(K, P), (r, g)
            assert np.array_equal(np.sort(got), want), (r, g)


def _q_rows(q, r, heads, G):
    return torch.cat([q[r, h * G:(h + 1) * G] for h in heads]).cpu()


def _run_decode(w, table, cache, seq_after, k1, v1, q, K):
    import query_aware_sparse_gb300 as qs
    gt = _table(table, seq_after)
    step = qs.DecodeStep(cache, gt, w.group, K)
    step(cache, gt, q, k1, v1)
    assert qs.device_error() == 0
    return step


def _gather(step, cache, r, heads, G):
    sl, sp, cnt = (np_of(x) for x in step.sel)
    out = np_of(step.out)[r]
    lse = np_of(step.lse)[r]
    rows = [h * G + x for h in heads for x in range(G)]
    return (np_of(cache.summary), np_of(step.scores), sl[r, heads], cnt[r, heads],
            out[rows], lse[rows])


def test_llama_layer_32k_fused_and_unfused():
    """Llama-2-7B-shaped layer, 32K context, budget 2048 (K = 128): the bench's step."""
    import query_aware_sparse_gb300 as qs
    w = wl.WORKLOADS["llama_layer"]
    L = int(w.lengths()[0])
    table = wl.make_page_table([L], w.page_size, seed=w.seed)
    k_tok, v_tok = wl.request_tokens(w, 0, L, device="cuda")
    q = wl.queries(w, [L - 1], device="cuda")
    cache = _gpu_cache(table, w)
    qs.append_kv(cache, _table(table, [L - 1]), k_tok[:L - 1].contiguous(),
                 v_tok[:L - 1].contiguous(), dev_i32([0, L - 1]), dev_i32([0]))
    twin = qs.PagedCache(cache.k_pool.clone(), cache.v_pool.clone(), cache.summary.clone())
    step = _run_decode(w, table, cache, [L], k_tok[L - 1:L].contiguous(),
                       v_tok[L - 1:L].contiguous(), q, w.k)
    heads = list(range(w.h_kv))              # every head: summaries, scores, sets, outputs
    unit = Unit(k_tok[:, heads].cpu(), v_tok[:, heads].cpu(), _q_rows(q, 0, heads, 1), heads, 1,
                w.page_size)
    ref = unit.oracle(L, w.k)
    gsum, gsc, gsel, gcnt, gout, glse = _gather(step, cache, 0, heads, 1)
    unit.check(ref, L, w.k, gsum, gsc[heads], gsel, gcnt, gout, glse, table.page_indices)
    check_every_selection(np_of(step.scores), np_of(step.sel[0]), np_of(step.sel[2]), table,
                          [L], w.k)
    # the unfused four calls on the twin cache give the same answer
    gt = _table(table, [L])
    qs.append_kv(twin, gt, k_tok[L - 1:L].contiguous(), v_tok[L - 1:L].contiguous(),
                 dev_i32([0, 1]), dev_i32([L - 1]))
    sc = qs.score_pages(twin, gt, q, 1)
    sl, sp, cnt = qs.select_topk(gt, w.h_kv, w.page_size, sc, w.k)
    o, lse = qs.sparse_decode_attn(twin, gt, q, 1, sl, sp, w.k)
    assert qs.device_error() == 0
    unit.check(ref, L, w.k, np_of(twin.summary), np_of(sc)[heads], np_of(sl)[0, heads],
               np_of(cnt)[0, heads], np_of(o)[0, heads], np_of(lse)[0, heads], table.page_indices)


def test_gqa_batch_16_requests_8k_to_128k():
    """16 ragged requests (8K..128K), 8 KV x 4 query heads, K = 256, permuted pool."""
    import query_aware_sparse_gb300 as qs
    w = wl.WORKLOADS["gqa_batch"]
    lens = w.lengths()
    table = wl.make_page_table(lens, w.page_size, seed=w.seed, permute=True, spare_pages=64)
    toks = [wl.request_tokens(w, r, int(L), device="cuda") for r, L in enumerate(lens)]
    pre = np.concatenate([[0], np.cumsum(lens - 1)]).astype(np.int32)
    kpre = torch.cat([k[:-1] for k, _ in toks]).contiguous()
    vpre = torch.cat([v[:-1] for _, v in toks]).contiguous()
    cache = _gpu_cache(table, w)
    qs.append_kv(cache, _table(table, lens - 1), kpre, vpre, dev_i32(pre),
                 dev_i32(np.zeros(len(lens))))
    del kpre, vpre
    k1 = torch.stack([k[-1] for k, _ in toks]).contiguous()
    v1 = torch.stack([v[-1] for _, v in toks]).contiguous()
    q = wl.queries(w, lens - 1, device="cuda")
    step = _run_decode(w, table, cache, lens, k1, v1, q, w.k)
    check_every_selection(np_of(step.scores), np_of(step.sel[0]), np_of(step.sel[2]), table,
                          lens, w.k)
    order = np.argsort(lens)
    heads = list(range(w.h_kv))              # every KV head of the sampled requests
    for r in (int(order[0]), int(order[len(order) // 2]), int(order[-1])):
        L = int(lens[r])
        k, v = toks[r]
        unit = Unit(k[:, heads].cpu(), v[:, heads].cpu(), _q_rows(q, r, heads, w.group), heads,
                    w.group, w.page_size)
        ref = unit.oracle(L, w.k)
        gsum, gsc, gsel, gcnt, gout, glse = _gather(step, cache, r, heads, w.group)
        lo = int(table.page_indptr[r])
        unit.check(ref, L, w.k, gsum, gsc[heads][:, lo:], gsel, gcnt, gout, glse,
                   table.page_indices[lo:])


def test_append_128k_prefill_then_64_decode_steps():
    """S = 32: prefill-append 131072 tokens, then 64 single-token decode steps."""
    import query_aware_sparse_gb300 as qs
    w = wl.WORKLOADS["append_128k"]
    L0 = int(w.lengths()[0])
    steps = w.decode_steps
    table = wl.make_page_table([L0 + steps], w.page_size, seed=w.seed)
    k_tok, v_tok = wl.request_tokens(w, 0, L0 + steps, device="cuda")
    cache = _gpu_cache(table, w)
    qs.append_kv(cache, _table(table, [L0]), k_tok[:L0].contiguous(), v_tok[:L0].contiguous(),
                 dev_i32([0, L0]), dev_i32([0]))
    assert qs.device_error() == 0
    heads = [0, 31]
    unit = Unit(k_tok[:, heads].cpu(), v_tok[:, heads].cpu(), torch.zeros(2, w.head_dim, dtype=w.dtype),
                heads, 1, w.page_size)
    ref0 = unit.oracle(L0, w.k)
    gs = np_of(cache.summary)[table.page_indices[:L0 // w.page_size]][:, heads]
    assert np.array_equal(gs.view(np.uint16), ref0["sm"][:L0 // w.page_size].view(np.uint16))
    gt_steps = None
    for s in range(steps):
        L = L0 + s + 1
        q = wl.queries(w, [L - 1], device="cuda", step=s)
        gt = _table(table, [L])
        if gt_steps is None:
            gt_steps = qs.DecodeStep(cache, gt, 1, w.k)
        gt_steps(cache, gt, q, k_tok[L - 1:L].contiguous(), v_tok[L - 1:L].contiguous())
        if s in (0, 31, steps - 1):
            assert qs.device_error() == 0
            unit.q = np_of(_q_rows(q, 0, heads, 1))
            ref = unit.oracle(L, w.k)
            gsum, gsc, gsel, gcnt, gout, glse = _gather(gt_steps, cache, 0, heads, 1)
            unit.check(ref, L, w.k, gsum, gsc[heads], gsel, gcnt, gout, glse, table.page_indices)
            check_every_selection(np_of(gt_steps.scores), np_of(gt_steps.sel[0]),
                                  np_of(gt_steps.sel[2]), table, [L], w.k)
    assert qs.device_error() == 0


def test_llama_32_layer_step_dense_and_budgets():
    """32 layers: layers 0-1 dense (K = P), layers 2-31 Quest with budgets
    1024 / 2048 / 4096 tokens in turn; layers 0, 1, 2, 3, 4 and 31 checked."""
    import query_aware_sparse_gb300 as qs
    w = wl.WORKLOADS["llama_step"]
    L = int(w.lengths()[0])
    P = -(-L // w.page_size)
    table = wl.make_page_table([L], w.page_size, seed=w.seed)
    heads = [3, 30]
    for layer in range(w.layers):
        K = P if layer < w.dense_layers else wl.selection_budget(
            w.budgets[(layer - w.dense_layers) % len(w.budgets)], w.page_size)
        k_tok, v_tok = wl.request_tokens(w, 0, L, layer=layer, device="cuda")
        q = wl.queries(w, [L - 1], layer=layer, device="cuda")
        cache = _gpu_cache(table, w)
        qs.append_kv(cache, _table(table, [L - 1]), k_tok[:L - 1].contiguous(),
                     v_tok[:L - 1].contiguous(), dev_i32([0, L - 1]), dev_i32([0]))
        step = _run_decode(w, table, cache, [L], k_tok[L - 1:L].contiguous(),
                           v_tok[L - 1:L].contiguous(), q, K)
        if layer in (0, 1, 2, 3, 4, w.layers - 1):
            unit = Unit(k_tok[:, heads].cpu(), v_tok[:, heads].cpu(), _q_rows(q, 0, heads, 1),
                        heads, 1, w.page_size)
            ref = unit.oracle(L, K)
            gsum, gsc, gsel, gcnt, gout, glse = _gather(step, cache, 0, heads, 1)
            unit.check(ref, L, K, gsum, gsc[heads], gsel, gcnt, gout, glse, table.page_indices)
            if layer < w.dense_layers:       # dense layer: plain attention over all tokens
                for j, h in enumerate(heads):
                    od, _ = qo.dense_attention(unit.q[j], unit.k[:, j], unit.v[:, j])
                    ok, rel = attn_close(gout[j][None], od[None])
                    assert ok.all(), rel
        del cache, step, k_tok, v_tok
