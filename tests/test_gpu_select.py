"""a3 parity: quest_select_topk against the oracle's sort on the same fp32
scores — integer output, so bit-exact (ids, physical ids, counts, order)."""

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quest_oracle as qo
from tests._cases import dev_i32, gpu_table, np_of

pytestmark = pytest.mark.gpu


def _select(lens, k, S, h_kv, scores, seed=0, reserve=0):
    import query_aware_sparse_gb300 as qs
    t = wl.make_page_table(lens, S, seed=seed, permute=True, spare_pages=5,
                           reserve_tokens=reserve)
    sc = torch.as_tensor(scores(t.nnz, h_kv), dtype=torch.float32)
    sl, sp, cnt = qs.select_topk(gpu_table(t), h_kv, S, sc.cuda(), k)
    assert qs.device_error() == 0
    ref = qo.select_topk(np_of(sc).astype(np.float64), t.page_indptr, t.page_indices, k)
    # oracle scores every table entry; restrict it to the scored pages
    for r in range(t.batch):
        P = -(-int(t.seq_lens[r]) // S)
        lo = int(t.page_indptr[r])
        for g in range(h_kv):
            chosen = qo.topk_pages(np_of(sc)[g, lo:lo + P].astype(np.float64), k)
            ref[0][r, g] = -1
            ref[1][r, g] = -1
            ref[0][r, g, :len(chosen)] = chosen
            ref[1][r, g, :len(chosen)] = t.page_indices[lo + chosen]
            ref[2][r, g] = len(chosen)
    return (np_of(sl), np_of(sp), np_of(cnt)), ref


def _gauss(seed):
    def f(n, h):
        g = torch.Generator().manual_seed(seed)
        return torch.randn((h, n), generator=g) * 30
    return f


def _ties(seed):
    def f(n, h):
        g = torch.Generator().manual_seed(seed)
        x = torch.randint(-3, 4, (h, n), generator=g).float()
        neg0 = torch.rand((h, n), generator=g) < 0.5
        x[(x == 0) & neg0] = -0.0
        return x
    return f


@pytest.mark.parametrize("gen", [_gauss, _ties])
@pytest.mark.parametrize("k", [1, 7, 8, 128, 300])
def test_select_matches_oracle(gen, k):
    lens = [1, 15, 16, 17, 1000, 16 * 128, 16 * 129 + 3, 5000, 0]
    got, ref = _select(lens, k, 16, 3, gen(k), seed=k)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_select_large_p_uses_global_path():
    lens = [16 * 20000 + 5, 16 * 16385]          # P = 20001 and 16385 > shared cache
    got, ref = _select(lens, 256, 16, 2, _ties(3), seed=9)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_select_reserved_entries_never_chosen():
    got, ref = _select([40, 500], 4, 32, 2, _gauss(4), seed=2, reserve=300)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_four_page_example(golden):
    import query_aware_sparse_gb300 as qs
    ex = golden("four_page_selection.json")
    table = qs.PageTable(dev_i32([0, 4]), dev_i32([3, 2, 1, 0]), dev_i32([64]))
    sc = torch.tensor([ex["U"]], dtype=torch.float32, device="cuda")
    for k, want in ex["selected"].items():
        sl, sp, cnt = qs.select_topk(table, 1, 16, sc, int(k))
        names = sorted(ex["pages"][i] for i in np_of(sl)[0, 0] if i >= 0)
        assert names == sorted(want)
        assert np_of(sp)[0, 0].tolist() == [3 - i for i in np_of(sl)[0, 0]]


# --------------------------------------------------------------------------
# Hybrid budget (local window + sink + Quest, Quest page §2.2 / §3.2)
# --------------------------------------------------------------------------

def _select_hybrid(lens, k, n_sink, n_local, S, h_kv, scores, seed=0, reserve=0):
    import query_aware_sparse_gb300 as qs
    t = wl.make_page_table(lens, S, seed=seed, permute=True, spare_pages=5,
                           reserve_tokens=reserve)
    sc = torch.as_tensor(scores(t.nnz, h_kv), dtype=torch.float32)
    sl, sp, cnt = qs.select_topk(gpu_table(t), h_kv, S, sc.cuda(), k,
                                 n_sink=n_sink, n_local=n_local)
    assert qs.device_error() == 0
    ref = qo.select_hybrid(np_of(sc).astype(np.float64), t.page_indptr, t.page_indices,
                           t.seq_lens, S, k, n_sink, n_local)
    return (np_of(sl), np_of(sp), np_of(cnt)), ref


@pytest.mark.parametrize("gen", [_gauss, _ties])
@pytest.mark.parametrize("k,n_sink,n_local", [(8, 1, 2), (128, 1, 32), (128, 0, 128),
                                              (300, 4, 0), (7, 7, 0), (16, 0, 5)])
def test_select_hybrid_matches_oracle(gen, k, n_sink, n_local):
    # short requests (sink and window overlap or cover everything), P < K and
    # P > K, a request long enough for the global-read path
    lens = [1, 15, 17, 40, 1000, 16 * 128, 16 * 129 + 3, 5000, 0]
    got, ref = _select_hybrid(lens, k, n_sink, n_local, 16, 3, gen(k + n_sink), seed=k)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_select_hybrid_page_budget_example():
    """The budget split of Quest page §2.2 at the llama_layer shape: 2048
    tokens = 32 local + 1 sink + 95 Quest pages over 2048 scored pages."""
    k, n_local, n_sink, quest = qo.hybrid_budget_pages(2048, 512, 4, 16)
    got, ref = _select_hybrid([32768], k, n_sink, n_local, 16, 4, _gauss(5), seed=3)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    sel = got[0][0, 0]
    assert sel[0] == 0 and list(sel[-n_local:]) == list(range(2048 - n_local, 2048))
    assert len(sel) == k == 1 + 32 + quest


def test_select_hybrid_large_p_uses_global_path():
    got, ref = _select_hybrid([16 * 20000 + 5], 256, 2, 40, 16, 2, _ties(6), seed=9)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
