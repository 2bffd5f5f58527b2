"""The C-ABI library builds, loads and exports every symbol include/quest.h
declares; host-side validation rejects bad arguments before any CUDA call.
No compute call is made here (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qlib():
    from query_aware_sparse_gb300 import build
    build.build()
    import query_aware_sparse_gb300 as q
    return q


def declared_symbols():
    with open(os.path.join(ROOT, "include", "quest.h")) as f:
        src = f.read()
    return set(re.findall(r"QUEST_API\s+[\w\s\*]+?\b(quest_\w+)\s*\(", src))


def test_header_declares_the_four_hot_path_calls():
    names = declared_symbols()
    for n in ("quest_append_kv", "quest_score_pages", "quest_select_topk",
              "quest_sparse_decode_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(qlib):
    L = qlib.lib()
    names = declared_symbols()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), n
    assert set(qlib.EXPORTED) == names


def test_status_strings(qlib):
    L = qlib.lib()
    assert L.quest_status_string(0) == b"QUEST_OK"
    for code in (-1, -2, -3, -4):
        assert L.quest_status_string(code).startswith(b"QUEST_ERR_")
    assert L.quest_status_string(99) == b"unknown quest_status"


def test_host_validation_rejects_bad_arguments(qlib):
    """These calls return before any CUDA call is made."""
    L = qlib.lib()
    C, Pg = qlib.QuestCache, qlib.QuestPages
    fake = 0x10000                      # never dereferenced: validation fails first
    good = C(fake, fake, fake, 8, 2, 16, 128, qlib.QUEST_F16)
    pages = Pg(fake, fake, fake, 1, 8)
    by = ctypes.byref
    # null cache / pools
    assert L.quest_append_kv(None, by(pages), fake, fake, 1, fake, fake, None) == -1
    assert L.quest_score_pages(by(C(0, fake, fake, 8, 2, 16, 128, 1)), by(pages), fake, 1, fake, None) == -1
    # unsupported head_dim / page_size / dtype / group
    assert L.quest_score_pages(by(C(fake, fake, fake, 8, 2, 16, 96, 1)), by(pages), fake, 1, fake, None) == -2
    assert L.quest_score_pages(by(C(fake, fake, fake, 8, 2, 24, 128, 1)), by(pages), fake, 1, fake, None) == -2
    assert L.quest_score_pages(by(C(fake, fake, fake, 8, 2, 16, 128, 7)), by(pages), fake, 1, fake, None) == -2
    assert L.quest_score_pages(by(good), by(pages), fake, 3, fake, None) == -2
    # misaligned pointers
    assert L.quest_score_pages(by(C(fake + 2, fake, fake, 8, 2, 16, 128, 1)), by(pages), fake, 1, fake, None) == -1
    assert L.quest_score_pages(by(good), by(pages), fake + 4, 1, fake, None) == -1
    # bad k / h_kv / page size for select
    assert L.quest_select_topk(by(pages), 2, 16, fake, 0, 0, 0, fake, fake, fake, None) == -1
    assert L.quest_select_topk(by(pages), 0, 16, fake, 4, 0, 0, fake, fake, fake, None) == -1
    assert L.quest_select_topk(by(pages), 2, 12, fake, 4, 0, 0, fake, fake, fake, None) == -2
    assert L.quest_select_topk(by(pages), 2, 16, fake, 4, 0, 0, None, fake, fake, None) == -1
    # hybrid budget: forced pages must be >= 0 and fit the budget
    assert L.quest_select_topk(by(pages), 2, 16, fake, 4, -1, 0, fake, fake, fake, None) == -1
    assert L.quest_select_topk(by(pages), 2, 16, fake, 4, 3, 2, fake, fake, fake, None) == -1
    # missing seq_lens where lengths are needed
    assert L.quest_select_topk(by(Pg(fake, fake, None, 1, 8)), 2, 16, fake, 4, 0, 0, fake, fake, fake, None) == -1
    # negative sizes
    assert L.quest_append_kv(by(good), by(pages), fake, fake, -1, fake, fake, None) == -1
    assert L.quest_append_kv(by(good), by(Pg(fake, fake, fake, -1, 8)), fake, fake, 1, fake, fake, None) == -1
    # attention: missing workspace is reported before any launch
    assert L.quest_sparse_decode_attn(by(good), by(pages), fake, 1, fake, fake, 4, fake, None,
                                      ctypes.c_float(0.0), None, 0, None) in (-3, -4)
    # E4M3 summaries: fp16 keys only, flag 0 or 1, not for the diagnostics
    f8_32 = C(fake, fake, fake, 8, 2, 16, 128, qlib.QUEST_F32, 1)
    assert L.quest_score_pages(by(f8_32), by(pages), fake, 1, fake, None) == -2
    assert L.quest_append_kv(by(f8_32), by(pages), fake, fake, 1, fake, fake, None) == -2
    assert L.quest_score_pages(by(C(fake, fake, fake, 8, 2, 16, 128, 1, 2)), by(pages), fake, 1,
                               fake, None) == -1
    f8 = C(fake, fake, fake, 8, 2, 16, 128, qlib.QUEST_F16, 1)
    assert L.quest_recall_diagnostics(by(f8), by(pages), fake, 1, fake, 4, 4, ctypes.c_float(0.0),
                                      fake, fake, fake, fake, fake, 1 << 20, None) == -2
    # per-head scores and the GQA union: the same validation as their relatives
    assert L.quest_score_pages_per_head(by(good), by(pages), fake, 3, fake, None) == -2
    assert L.quest_score_pages_per_head(by(good), by(pages), fake + 4, 1, fake, None) == -1
    assert L.quest_union_decode_attn(by(good), by(pages), fake, 4, fake, 0, fake, None,
                                     ctypes.c_float(0.0), fake, fake, fake, fake, 1 << 20,
                                     None) == -1
    assert L.quest_union_decode_attn(by(good), by(pages), fake, 4, None, 8, fake, None,
                                     ctypes.c_float(0.0), fake, fake, fake, fake, 1 << 20,
                                     None) == -1
    assert L.quest_union_workspace_size(1, 2, 3, 128, 16, qlib.QUEST_F16, 8) == 0
    # empty batches are valid no-ops
    empty = Pg(None, None, None, 0, 0)
    assert L.quest_select_topk(by(empty), 2, 16, None, 4, 0, 0, None, None, None, None) == 0
    assert L.quest_append_kv(by(good), by(empty), None, None, 0, None, None, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import query_aware_sparse_gb300 as q
    monkeypatch.setattr(q, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(q, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        q.lib()


def test_workspace_sizes_host_logic(qlib):
    """Workspace sizing is host logic (no GPU needed): closed forms and the
    relations between the calls."""
    L = qlib.lib()
    up = lambda b: (b + 255) // 256 * 256
    # diagnostics: token logits, per-page softmax statistics, per-page |v| maxima
    for h, G, nnz, S in ((32, 1, 2048, 16), (8, 4, 70000, 16), (2, 8, 5, 32)):
        want = up(h * G * nnz * S * 4) + up(h * G * nnz * 8) + up(h * nnz * 4)
        assert L.quest_diag_workspace_size(h, G, nnz, S) == want
    assert L.quest_diag_workspace_size(2, 3, 5, 16) == 0
    # union: its physical ids, then the split-K partials of G*k slots
    for B, h, G, d, S, k in ((16, 8, 4, 128, 16, 256), (1, 2, 2, 64, 32, 7), (3, 4, 8, 128, 16, 9)):
        ws = L.quest_union_workspace_size(B, h, G, d, S, qlib.QUEST_F16, k)
        phys = up(B * h * G * k * 4)
        attn = L.quest_attn_workspace_size(B, h, G, d, S, G * k)
        assert phys < ws <= phys + attn
    assert L.quest_union_workspace_size(1, 2, 4, 96, 16, qlib.QUEST_F16, 8) == 0
    # attention and the fused step: positive for supported shapes, 0 otherwise
    assert L.quest_attn_workspace_size(1, 32, 1, 128, 16, 128) > 0
    assert L.quest_attn_workspace_size(1, 32, 3, 128, 16, 128) == 0
    assert L.quest_decode_workspace_size(1, 2048, 32, 1, 128, 16, qlib.QUEST_F16, 128) > 0
    assert L.quest_decode_workspace_size(1, 2048, 32, 1, 96, 16, qlib.QUEST_F16, 128) == 0
    assert L.quest_decode_workspace_size(1, 2048, 32, 1, 128, 24, qlib.QUEST_F16, 128) == 0


def test_decode_step_kernel_choice_host_logic(qlib):
    """Which kernel quest_decode_step takes is host logic: the cluster kernel
    for groups 1 and 2 (and 4 and 8 with fp16 K/V) while the (request, KV
    head) units fit 64 per cluster, the grid-wide kernel otherwise, 0 for
    unsupported shapes. With no device the plan assumes 32 resident
    clusters."""
    L = qlib.lib()
    F16, F32 = qlib.QUEST_F16, qlib.QUEST_F32
    assert L.quest_decode_step_kernel(1, 32, 1, 128, 16, F16, 128, 0) == 2
    assert L.quest_decode_step_kernel(16, 8, 4, 128, 16, F16, 256, 0) == 2
    assert L.quest_decode_step_kernel(3, 2, 8, 64, 32, F16, 8, 1) == 2
    assert L.quest_decode_step_kernel(2, 4, 2, 64, 16, F32, 8, 0) == 2
    assert L.quest_decode_step_kernel(2, 4, 4, 64, 16, F32, 8, 0) == 1    # fp32 GQA of 4
    assert L.quest_decode_step_kernel(64 * 32, 1, 1, 64, 16, F16, 8, 0) == 2   # 64 per cluster
    assert L.quest_decode_step_kernel(64 * 32 + 1, 1, 1, 64, 16, F16, 8, 0) == 1
    assert L.quest_decode_step_kernel(1, 32, 3, 128, 16, F16, 128, 0) == 0
    assert L.quest_decode_step_kernel(1, 32, 1, 96, 16, F16, 128, 0) == 0
    assert L.quest_decode_step_kernel(1, 32, 1, 128, 16, F32, 128, 1) == 0  # E4M3 needs fp16
    # the cluster kernel keeps everything in shared memory: a nominal workspace
    assert L.quest_decode_workspace_size(1, 2048, 32, 1, 128, 16, F16, 128) == 256
