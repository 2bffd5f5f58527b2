"""Shared builders for the GPU parity tests: seeded inputs from ``workloads``,
the same stored tensors handed to the CUDA path (device) and to the oracle
(host numpy copies). Holds no arithmetic of the method."""

from __future__ import annotations

import math

import numpy as np
import torch

import workloads as wl

F16 = torch.float16
F32 = torch.float32


def np_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def dev_i32(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device="cuda")


def random_case(seed, lens, *, h_kv=2, group=1, d=64, S=16, dtype=F16,
                permute=True, spare=3, reserve_tokens=0, scale=1.0,
                signed_zeros=False):
    """A ragged batch laid out in a NaN-poisoned pool (host tensors)."""
    table = wl.make_page_table(lens, S, seed=seed, permute=permute,
                               spare_pages=spare, reserve_tokens=reserve_tokens)
    g = torch.Generator().manual_seed(seed)
    n = int(np.sum(lens))
    k = (torch.randn((n, h_kv, d), generator=g) * scale).to(dtype)
    v = torch.randn((n, h_kv, d), generator=g).to(dtype)
    if signed_zeros and n:
        z = torch.rand((n, h_kv, d), generator=g) < 0.05
        sgn = torch.rand((n, h_kv, d), generator=g) < 0.5
        k[z & sgn] = 0.0
        k[z & ~sgn] = -0.0
    q = torch.randn((len(lens), h_kv * group, d), generator=g).to(dtype)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    kp, vp, sm = wl.empty_pool(table, h_kv, d, dtype)
    wl.place_tokens(kp, table, k, indptr)
    wl.place_tokens(vp, table, v, indptr)
    return dict(table=table, k_tok=k, v_tok=v, q=q, k_pool=kp, v_pool=vp,
                summary=sm, tok_indptr=indptr, h_kv=h_kv, group=group, d=d, S=S,
                dtype=dtype)


def gpu_table(table: wl.PageTable, seq_lens=None):
    import query_aware_sparse_gb300 as qs
    sl = table.seq_lens if seq_lens is None else seq_lens
    return qs.PageTable(dev_i32(table.page_indptr), dev_i32(table.page_indices),
                        dev_i32(sl), nnz=table.nnz)


def gpu_cache(k_pool, v_pool, summary):
    import query_aware_sparse_gb300 as qs
    return qs.PagedCache(k_pool.cuda().contiguous(), v_pool.cuda().contiguous(),
                         summary.cuda().contiguous())


def score_tol(q, summary_np, table, group):
    """1e-4 * sum_j |q_j| max(|m_j|, |M_j|) per (KV head, entry), maximised
    over the group's query heads."""
    qn = np.abs(np.asarray(q, dtype=np.float64))
    h_kv = summary_np.shape[1]
    tol = np.zeros((h_kv, table.nnz))
    for r in range(table.batch):
        lo, hi = int(table.page_indptr[r]), int(table.page_indptr[r + 1])
        phys = table.page_indices[lo:hi]
        mag = np.maximum(np.abs(summary_np[phys, :, 0].astype(np.float64)),
                         np.abs(summary_np[phys, :, 1].astype(np.float64)))   # [P, h_kv, d]
        for gk in range(h_kv):
            heads = range(gk * group, (gk + 1) * group)
            tol[gk, lo:hi] = 1e-4 * np.max([mag[:, gk] @ qn[r, h] for h in heads], axis=0)
    return tol


def attn_close(o_gpu, o_ref, rel=2e-3):
    """Row-max-relative check: max_j |o - ref| <= rel * max(max_j |ref|, 1e-6)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o_gpu - o_ref).max(axis=-1)
    den = np.maximum(np.abs(o_ref).max(axis=-1), 1e-6)
    return err <= rel * den, err / den


def check_selection(sel_gpu, cnt_gpu, scores_ref, tol, table, k, rows, n_sink=0, n_local=0):
    """GPU sets equal the oracle's except pages whose oracle score lies within
    the score tolerance of the oracle's last Quest score; forced pages (hybrid
    budget: first n_sink, last n_local) always present; no duplicates; counts."""
    from oracle import quest_oracle as qo
    for (r, g) in rows:
        lo = int(table.page_indptr[r])
        P = -(-int(table.seq_lens[r]) // table.page_size)
        U = scores_ref[g, lo:lo + P]
        forced = set(qo.forced_pages(P, n_sink, n_local))
        want = set(qo.hybrid_pages(U, P, k, n_sink, n_local).tolist())
        got_list = [int(x) for x in sel_gpu[r, g] if x >= 0]
        got = set(got_list)
        assert len(got) == len(got_list), "duplicate page ids"
        assert int(cnt_gpu[r, g]) == min(k, P) == len(got)
        assert forced <= got, (r, g, sorted(forced - got))
        if P <= k:
            assert got == set(range(P))
            continue
        kq = k - len(forced)                 # Quest's share of the budget
        if kq == 0:
            assert got == forced
            continue
        rest = np.array([U[i] for i in range(P) if i not in forced])
        kth = np.sort(rest)[::-1][kq - 1]
        for p in got ^ want:
            assert p not in forced
            assert abs(U[p] - kth) <= tol[g, lo + p] + 1e-12, (r, g, p, U[p], kth)


def default_scale(d):
    return 1.0 / math.sqrt(d)
