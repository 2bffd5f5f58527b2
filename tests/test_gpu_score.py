"""a2 parity: quest_score_pages against the oracle's fp64 eq (2)-(3) bound,
within 1e-4 * sum_j |q_j| max(|m_j|, |M_j|)."""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import F16, F32, gpu_cache, gpu_table, np_of, random_case, score_tol

pytestmark = pytest.mark.gpu


def _score_case(case):
    import query_aware_sparse_gb300 as qs
    t = case["table"]
    osm = qo.build_summary(np_of(case["k_pool"]), t.page_indptr, t.page_indices, t.seq_lens,
                           summary=np_of(case["summary"]).copy())
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(osm))
    table = gpu_table(t)
    sc = qs.score_pages(cache, table, case["q"].cuda(), case["group"])
    assert qs.device_error() == 0
    ref = qo.score_pages(np_of(case["q"]), osm, t.page_indptr, t.page_indices, case["group"])
    return np_of(sc), ref, osm


@pytest.mark.parametrize("dtype,d,group", [(F16, 128, 1), (F16, 128, 4), (F16, 64, 2),
                                           (F32, 64, 1), (F32, 128, 8), (F16, 64, 8)])
def test_scores_match_oracle(dtype, d, group):
    lens = [1, 15, 16, 17, 250, 1000, 33]
    case = random_case(21 + d + group, lens, h_kv=3, group=group, d=d, S=16,
                       dtype=dtype, scale=2.0, signed_zeros=True)
    got, ref, osm = _score_case(case)
    tol = score_tol(np_of(case["q"]), osm, case["table"], group)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)


@pytest.mark.parametrize("group,S", [(1, 32), (4, 32), (8, 16)])
def test_reserved_entries_score_minus_inf(group, S):
    # groups of 4 and 8 take the warp-MMA bound; chunks of 8 table entries
    # there span requests and reserved entries
    case = random_case(31 + group, [40, 3, 77, 1, 200], h_kv=2, group=group, d=128, S=S,
                       reserve_tokens=70)
    got, ref, osm = _score_case(case)
    t = case["table"]
    tol = score_tol(np_of(case["q"]), osm, t, group)
    for r in range(t.batch):
        lo, hi = t.page_indptr[r], t.page_indptr[r + 1]
        P = -(-int(t.seq_lens[r]) // S)
        assert np.all(got[:, lo + P:hi] == -np.inf)
        assert np.all(np.abs(got[:, lo:lo + P] - ref[:, lo:lo + P]) <= tol[:, lo:lo + P])


def test_worked_example_embedded():
    """The Quest page §1.1 example in d=64 (zeros elsewhere add nothing)."""
    import query_aware_sparse_gb300 as qs
    from tests._cases import dev_i32
    d = 64
    keys = torch.zeros((3, 1, d), dtype=F32)
    keys[:, 0, :2] = torch.tensor([[1., 4.], [3., -2.], [-1., 1.]])
    q = torch.zeros((1, 1, d), dtype=F32)
    q[0, 0, :2] = torch.tensor([2., -1.])
    kp = torch.zeros((1, 1, 16, d), device="cuda")
    cache = qs.PagedCache(kp, torch.zeros_like(kp), torch.zeros((1, 1, 2, d), device="cuda"))
    table = qs.PageTable(dev_i32([0, 1]), dev_i32([0]), dev_i32([3]))
    qs.append_kv(cache, table, keys.cuda(), keys.cuda(), dev_i32([0, 3]), dev_i32([0]))
    sm = np_of(cache.summary)[0, 0]
    assert sm[0, :2].tolist() == [-1, -2] and sm[1, :2].tolist() == [3, 4]
    assert np_of(qs.score_pages(cache, table, q.cuda(), 1))[0, 0] == 8.0
