"""a4/a5 parity: quest_sparse_decode_attn against the oracle's fp64
attention over the same page sets, within 2e-3 row-max-relative error;
padding slots are NaN-poisoned, so any read of them shows up."""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import (F16, F32, attn_close, dev_i32, gpu_cache, gpu_table, np_of,
                          random_case)

pytestmark = pytest.mark.gpu


def _sets(case, k, mode, seed):
    """Page sets [B, h_kv, k] (logical, physical), -1 padded."""
    t = case["table"]
    rng = np.random.default_rng(seed)
    B, h = t.batch, case["h_kv"]
    sl = np.full((B, h, k), -1, np.int32)
    for r in range(B):
        P = -(-int(t.seq_lens[r]) // t.page_size)
        for g in range(h):
            if mode == "all":
                ch = np.arange(min(P, k))
            elif mode == "random":
                n = int(rng.integers(0, min(P, k) + 1))
                ch = rng.choice(P, size=n, replace=False) if n else np.zeros(0, int)
            elif mode == "tail":
                ch = np.array([P - 1]) if P else np.zeros(0, int)
            slots = rng.permutation(k)[:len(ch)] if mode == "random" else np.arange(len(ch))
            sl[r, g, slots] = ch
    sp = np.where(sl >= 0, t.page_indices[np.maximum(sl, 0) + t.page_indptr[:-1, None, None]], -1)
    return sl, sp.astype(np.int32)


def _attn(case, k, mode, seed=0):
    import query_aware_sparse_gb300 as qs
    t = case["table"]
    sl, sp = _sets(case, k, mode, seed)
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    o, lse = qs.sparse_decode_attn(cache, gpu_table(t), case["q"].cuda(), case["group"],
                                   dev_i32(sl), dev_i32(sp), k)
    assert qs.device_error() == 0
    ro, rl = qo.sparse_attention(np_of(case["q"]), np_of(case["k_pool"]), np_of(case["v_pool"]),
                                 t.page_indptr, t.page_indices, t.seq_lens, sl, case["group"])
    return np_of(o), np_of(lse), ro, rl


CONFIGS = [(F16, 128, 16, 1), (F16, 128, 16, 4), (F16, 64, 32, 2), (F32, 64, 16, 1),
           (F16, 128, 32, 1), (F16, 128, 16, 8), (F32, 128, 16, 2)]


@pytest.mark.parametrize("dtype,d,S,group", CONFIGS)
@pytest.mark.parametrize("mode", ["all", "random", "tail"])
def test_attention_matches_oracle(dtype, d, S, group, mode):
    lens = [1, 15, 16, 17, 200, 1000, 0, 3 * S]
    case = random_case(40 + d + S + group, lens, h_kv=2, group=group, d=d, S=S, dtype=dtype)
    k = 40
    o, lse, ro, rl = _attn(case, k, mode, seed=d + group)
    empty = ~np.isfinite(rl)
    assert np.all(o[empty] == 0) and np.all(lse[empty] == -np.inf)
    ok, rel = attn_close(o[~empty], ro[~empty])
    assert ok.all(), rel.max()
    assert np.all(np.abs(lse[~empty] - rl[~empty]) <= 1e-3 * np.maximum(1, np.abs(rl[~empty])))


def test_all_pages_equals_dense_attention():
    """K = P: the selection covers every page, so the result is dense attention
    over the contiguous, un-paged tokens (Quest page §1.2, dense fallback)."""
    import query_aware_sparse_gb300 as qs
    lens = [300, 17, 1]
    case = random_case(5, lens, h_kv=2, group=2, d=128, S=16)
    t = case["table"]
    o, lse, _, _ = _attn(case, 19, "all")
    for r, L in enumerate(lens):
        a, b = case["tok_indptr"][r], case["tok_indptr"][r + 1]
        for h in range(4):
            od, _ = qo.dense_attention(np_of(case["q"])[r, h], np_of(case["k_tok"])[a:b, h // 2],
                                       np_of(case["v_tok"])[a:b, h // 2])
            ok, rel = attn_close(o[r, h][None], od[None])
            assert ok.all(), rel


def test_page_order_and_physical_shuffle_invariance():
    import query_aware_sparse_gb300 as qs
    case = random_case(8, [700], h_kv=1, d=128, S=16)
    t = case["table"]
    sl, sp = _sets(case, 12, "random", 3)
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    tab = gpu_table(t)
    q = case["q"].cuda()
    o1, _ = qs.sparse_decode_attn(cache, tab, q, 1, dev_i32(sl), dev_i32(sp), 12)
    perm = np.random.default_rng(1).permutation(12)
    o2, _ = qs.sparse_decode_attn(cache, tab, q, 1, dev_i32(sl[..., perm]), dev_i32(sp[..., perm]), 12)
    ok, rel = attn_close(np_of(o1), np_of(o2), rel=1e-5)
    assert ok.all(), rel


def test_bad_page_id_is_reported_and_skipped():
    import query_aware_sparse_gb300 as qs
    case = random_case(9, [64], h_kv=1, d=64, S=16)
    t = case["table"]
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    sl = np.array([[[0, 1]]], np.int32)
    sp = np.array([[[t.page_indices[0], 10 ** 6]]], np.int32)
    o, _ = qs.sparse_decode_attn(cache, gpu_table(t), case["q"].cuda(), 1,
                                 dev_i32(sl), dev_i32(sp), 2)
    assert qs.device_error() & 1
    ro, _ = qo.sparse_attention(np_of(case["q"]), np_of(case["k_pool"]), np_of(case["v_pool"]),
                                t.page_indptr, t.page_indices, t.seq_lens,
                                np.array([[[0, -1]]], np.int32), 1)
    ok, rel = attn_close(np_of(o), ro)
    assert ok.all()
