"""E4M3 page summaries with directed rounding (Quest page §3, the paragraph
on the summary dtype) through quest_append_kv and quest_score_pages: codes
bit-exact against the oracle's rounding of the exact summary (also when a
page is filled over several appends, the codes being folded in place), and
scores within 1e-4 * sum_j |q_j| max(|m8_j|, |M8_j|) of the oracle's fp64
bound over the decoded box."""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import F16, dev_i32, gpu_table, np_of, random_case, score_tol

pytestmark = pytest.mark.gpu


def _append_in_chunks(cache, table, case, chunks):
    """Append each request's tokens in `chunks` slices (ragged boundaries)."""
    import query_aware_sparse_gb300 as qs
    t = case["table"]
    lens = np.asarray(t.seq_lens)
    B = len(lens)
    cuts = [np.linspace(0, L, chunks + 1).astype(np.int64) for L in lens]
    for c in range(chunks):
        before = np.array([cuts[r][c] for r in range(B)], np.int32)
        after = np.array([cuts[r][c + 1] for r in range(B)], np.int32)
        rows = np.concatenate([np.arange(case["tok_indptr"][r] + before[r],
                                         case["tok_indptr"][r] + after[r]) for r in range(B)])
        kn = case["k_tok"][rows].contiguous().cuda()
        vn = case["v_tok"][rows].contiguous().cuda()
        ind = np.concatenate([[0], np.cumsum(after - before)]).astype(np.int32)
        qs.append_kv(cache, gpu_table(t, seq_lens=after), kn, vn, dev_i32(ind), dev_i32(before))
    assert qs.device_error() == 0


@pytest.mark.parametrize("d,S,group,chunks", [(128, 16, 1, 1), (128, 16, 4, 3), (64, 32, 2, 5),
                                              (64, 16, 8, 2)])
def test_append_and_score_e4m3(d, S, group, chunks):
    import query_aware_sparse_gb300 as qs
    lens = [1, 15, 16, 17, 250, 1000, 33]
    case = random_case(70 + d + S + group + chunks, lens, h_kv=3, group=group, d=d, S=S,
                       dtype=F16, scale=3.0, signed_zeros=True)
    t = case["table"]
    sm8 = torch.full(case["summary"].shape, 0x7F, dtype=torch.uint8, device="cuda")
    cache = qs.PagedCache(case["k_pool"].cuda().contiguous(),
                          torch.zeros_like(case["v_pool"]).cuda(), sm8)
    cache.k_pool.fill_(float("nan"))
    _append_in_chunks(cache, t, case, chunks)
    exact = qo.build_summary(np_of(case["k_pool"]), t.page_indptr, t.page_indices, t.seq_lens)
    want, ovf = qo.summary_to_e4m3(exact)
    assert not ovf.any()
    got = np_of(cache.summary)
    for r in range(t.batch):
        P = -(-int(t.seq_lens[r]) // S)
        phys = t.page_indices[t.page_indptr[r]:t.page_indptr[r] + P]
        assert np.array_equal(got[phys], want[phys]), r
    q = case["q"]
    sc = np_of(qs.score_pages(cache, gpu_table(t), q.cuda(), group))
    assert qs.device_error() == 0
    ref = qo.score_pages_e4m3(np_of(q), want, t.page_indptr, t.page_indices, group)
    tol = score_tol(np_of(q), qo.e4m3_decode(want), t, group)
    exact_ref = qo.score_pages(np_of(q), exact, t.page_indptr, t.page_indices, group)
    for r in range(t.batch):
        lo = t.page_indptr[r]
        P = -(-int(t.seq_lens[r]) // S)
        assert np.all(np.abs(sc[:, lo:lo + P] - ref[:, lo:lo + P]) <= tol[:, lo:lo + P])
        # the rounded-out box never scores below the exact one (eq (4) kept)
        assert np.all(sc[:, lo:lo + P] >= exact_ref[:, lo:lo + P] - tol[:, lo:lo + P])
        assert np.all(sc[:, lo + P:t.page_indptr[r + 1]] == -np.inf)


def test_worked_example_e4m3():
    """The Quest page §1.1 example: its box is on the E4M3 grid, U stays 8."""
    import query_aware_sparse_gb300 as qs
    d = 64
    keys = torch.zeros((3, 1, d), dtype=F16)
    keys[:, 0, :2] = torch.tensor([[1., 4.], [3., -2.], [-1., 1.]], dtype=F16)
    q = torch.zeros((1, 1, d), dtype=F16)
    q[0, 0, :2] = torch.tensor([2., -1.], dtype=F16)
    kp = torch.zeros((1, 1, 16, d), dtype=F16, device="cuda")
    cache = qs.PagedCache(kp, torch.zeros_like(kp),
                          torch.zeros((1, 1, 2, d), dtype=torch.uint8, device="cuda"))
    table = qs.PageTable(dev_i32([0, 1]), dev_i32([0]), dev_i32([3]))
    qs.append_kv(cache, table, keys.cuda(), keys.cuda(), dev_i32([0, 3]), dev_i32([0]))
    codes = np_of(cache.summary)[0, 0]
    assert qo.e4m3_decode(codes[0, :2]).tolist() == [-1.0, -2.0]
    assert qo.e4m3_decode(codes[1, :2]).tolist() == [3.0, 4.0]
    assert np_of(qs.score_pages(cache, table, q.cuda(), 1))[0, 0] == 8.0


def test_keys_beyond_448_are_flagged():
    """A key outside +-448 has no E4M3 bound on its far side: the code
    saturates and the device error word says so (no fault, no trap)."""
    import query_aware_sparse_gb300 as qs
    d = 64
    keys = torch.zeros((2, 1, d), dtype=F16)
    keys[0, 0, 0] = 1000.0
    keys[1, 0, 1] = -500.0
    kp = torch.zeros((1, 1, 16, d), dtype=F16, device="cuda")
    cache = qs.PagedCache(kp, torch.zeros_like(kp),
                          torch.zeros((1, 1, 2, d), dtype=torch.uint8, device="cuda"))
    table = qs.PageTable(dev_i32([0, 1]), dev_i32([0]), dev_i32([2]))
    qs.append_kv(cache, table, keys.cuda(), keys.cuda(), dev_i32([0, 2]), dev_i32([0]))
    assert qs.device_error() == 0x10
    codes = np_of(cache.summary)[0, 0]
    exact = qo.build_summary(np_of(cache.k_pool), np.array([0, 1]), np.array([0]), np.array([2]))
    want, ovf = qo.summary_to_e4m3(exact)
    assert ovf.any()
    assert np.array_equal(codes, want[0, 0])
