"""query_aware_sparse_gb300 — Quest-style query-aware page selection on GB300.

A thin Python binding over ``libquest.so`` (the C ABI in ``include/quest.h``).
Every function here only marshals arguments (tensor data pointers, sizes and
the current CUDA stream) and calls the library; all the computation runs in
the library's CUDA kernels. There is no fallback: if the library is missing or
a call fails, an exception is raised.

Tensors are torch tensors on the current CUDA device (torch is used for device
memory and streams only).
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libquest.so")

QUEST_F32, QUEST_F16 = 0, 1
DEVERR = {1: "page id outside the pool", 2: "beyond the page table",
          4: "selected page holds no valid token", 8: "in-kernel wait timed out",
          16: "key beyond +-448 under an E4M3 summary"}


class QuestCache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("summary", ctypes.c_void_p), ("n_phys", ctypes.c_int32),
                ("h_kv", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("summary_fp8", ctypes.c_int32)]


class QuestPages(ctypes.Structure):
    _fields_ = [("page_indptr", ctypes.c_void_p), ("page_indices", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("nnz", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libquest.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m query_aware_sparse_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.quest_append_kv.argtypes = [P, P, P, P, I32, P, P, P]
        L.quest_score_pages.argtypes = [P, P, P, I32, P, P]
        L.quest_score_pages_per_head.argtypes = [P, P, P, I32, P, P]
        L.quest_union_decode_attn.argtypes = [P, P, P, I32, P, I32, P, P, ctypes.c_float, P, P,
                                              P, P, SZ, P]
        L.quest_union_decode_attn.restype = I32
        L.quest_union_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, I32]
        L.quest_union_workspace_size.restype = SZ
        L.quest_select_topk.argtypes = [P, I32, I32, P, I32, I32, I32, P, P, P, P]
        L.quest_sparse_decode_attn.argtypes = [P, P, P, I32, P, P, I32, P, P,
                                               ctypes.c_float, P, SZ, P]
        L.quest_sparse_decode_attn_noalloc.argtypes = [P, P, P, I32, P, P, I32, P, P,
                                                       ctypes.c_float, P]
        L.quest_sparse_decode_attn_noalloc.restype = I32
        L.quest_attn_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32]
        L.quest_attn_workspace_size.restype = SZ
        L.quest_decode_step.argtypes = [P, P, P, P, P, I32, I32, I32, I32, P, P, P, P, P, P,
                                        ctypes.c_float, P, SZ, P]
        L.quest_decode_step.restype = I32
        L.quest_decode_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32]
        L.quest_decode_workspace_size.restype = SZ
        L.quest_decode_step_kernel.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32]
        L.quest_decode_step_kernel.restype = I32
        L.quest_recall_diagnostics.argtypes = [P, P, P, I32, P, I32, I32, ctypes.c_float, P, P,
                                               P, P, P, SZ, P]
        L.quest_recall_diagnostics.restype = I32
        L.quest_diag_workspace_size.argtypes = [I32, I32, I32, I32]
        L.quest_diag_workspace_size.restype = SZ
        L.quest_set_trace.argtypes = [P, I32, I32, I32, I32, I32, I32, I32, I32]
        L.quest_set_trace.restype = I32
        L.quest_test_step_fault.argtypes = [I32, I32]
        L.quest_test_step_fault.restype = I32
        L.quest_get_device_error.argtypes = [P]
        L.quest_get_device_error.restype = I32
        L.quest_status_string.argtypes = [I32]
        L.quest_status_string.restype = ctypes.c_char_p
        for fn in ("quest_append_kv", "quest_score_pages", "quest_select_topk",
                   "quest_sparse_decode_attn"):
            getattr(L, fn).restype = I32
        _lib = L
    return _lib


EXPORTED = ("quest_append_kv", "quest_score_pages", "quest_score_pages_per_head",
            "quest_select_topk", "quest_union_decode_attn", "quest_union_workspace_size",
            "quest_sparse_decode_attn", "quest_sparse_decode_attn_noalloc",
            "quest_attn_workspace_size",
            "quest_decode_step", "quest_decode_workspace_size", "quest_decode_step_kernel",
            "quest_recall_diagnostics", "quest_diag_workspace_size", "quest_set_trace",
            "quest_test_step_fault", "quest_get_device_error", "quest_status_string")


def _check(status: int) -> None:
    if status != 0:
        raise RuntimeError(lib().quest_status_string(status).decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return QUEST_F16
    if dt == torch.float32:
        return QUEST_F32
    raise ValueError(f"unsupported element type {dt}")


class PagedCache:
    """One layer's pool + summary (caller-owned torch tensors).

    k_pool, v_pool: [n_phys, h_kv, page_size, head_dim]; summary:
    [n_phys, h_kv, 2, head_dim] (index 0 = min, 1 = max), either in the K/V
    dtype or, as a torch.uint8 tensor, E4M3 codes with directed rounding
    (fp16 K/V only; see summary_fp8 in quest.h).
    """

    def __init__(self, k_pool, v_pool, summary):
        self.k_pool, self.v_pool, self.summary = k_pool, v_pool, summary
        n_phys, h_kv, S, d = k_pool.shape
        self.n_phys, self.h_kv, self.page_size, self.head_dim = n_phys, h_kv, S, d
        self.dtype = k_pool.dtype
        self.summary_fp8 = summary.dtype == torch.uint8
        if not self.summary_fp8 and summary.dtype != k_pool.dtype:
            raise ValueError("summary must have the K/V dtype or be uint8 E4M3 codes")
        self.c = QuestCache(k_pool.data_ptr(), v_pool.data_ptr(), summary.data_ptr(),
                            n_phys, h_kv, S, d, dtype_code(k_pool.dtype), int(self.summary_fp8))

    @classmethod
    def empty(cls, n_phys, h_kv, page_size, head_dim, dtype, device="cuda", summary_fp8=False):
        kp = torch.empty((n_phys, h_kv, page_size, head_dim), dtype=dtype, device=device)
        vp = torch.empty_like(kp)
        sm = torch.empty((n_phys, h_kv, 2, head_dim), dtype=torch.uint8 if summary_fp8 else dtype,
                         device=device)
        return cls(kp, vp, sm)


class PageTable:
    """Ragged page table on the device: page_indptr [B+1], page_indices [nnz],
    seq_lens [B] (int32). ``nnz`` is kept on the host."""

    def __init__(self, page_indptr, page_indices, seq_lens, nnz=None):
        self.page_indptr, self.page_indices, self.seq_lens = page_indptr, page_indices, seq_lens
        self.batch = int(seq_lens.shape[0])
        self.nnz = int(page_indices.shape[0]) if nnz is None else int(nnz)
        self.c = QuestPages(page_indptr.data_ptr(), page_indices.data_ptr(),
                            seq_lens.data_ptr(), self.batch, self.nnz)


def append_kv(cache: PagedCache, table: PageTable, k_new, v_new, append_indptr,
              seq_lens_before, stream=None) -> None:
    """quest_append_kv: write k_new/v_new [n_new, h_kv, d] into the pool and
    update the page min/max summaries."""
    _check(lib().quest_append_kv(ctypes.byref(cache.c), ctypes.byref(table.c),
                                 _ptr(k_new), _ptr(v_new), int(k_new.shape[0]),
                                 _ptr(append_indptr), _ptr(seq_lens_before),
                                 _stream(stream)))


def score_pages(cache: PagedCache, table: PageTable, q, group: int, scores=None,
                stream=None):
    """quest_score_pages: scores [h_kv, nnz] fp32 of every page-table entry."""
    if scores is None:
        scores = torch.empty((cache.h_kv, table.nnz), dtype=torch.float32, device=q.device)
    _check(lib().quest_score_pages(ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q),
                                   int(group), _ptr(scores), _stream(stream)))
    return scores


def score_pages_per_head(cache: PagedCache, table: PageTable, q, group: int, scores=None,
                         stream=None):
    """quest_score_pages_per_head: scores [h_kv * group, nnz] fp32, one row per
    query head (no group max)."""
    if scores is None:
        scores = torch.empty((cache.h_kv * group, table.nnz), dtype=torch.float32, device=q.device)
    _check(lib().quest_score_pages_per_head(ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q),
                                            int(group), _ptr(scores), _stream(stream)))
    return scores


def union_workspace_size(batch, h_kv, group, head_dim, page_size, dtype, k) -> int:
    return int(lib().quest_union_workspace_size(batch, h_kv, group, head_dim, page_size,
                                                dtype_code(dtype), k))


def union_decode_attn(cache: PagedCache, table: PageTable, q, group: int, sel_logical, k: int,
                      out=None, lse=None, sm_scale: float = 0.0, union=None, workspace=None,
                      stream=None):
    """quest_union_decode_attn: per-query-head page sets sel_logical
    [B, h_q, k]; returns (out [B, h_q, d], lse [B, h_q], (union_logical
    [B, h_kv, group * k], union_mask uint8 [B, h_kv, group * k], union_count
    [B, h_kv]))."""
    B, h_q, d = q.shape
    dev = q.device
    h_kv = cache.h_kv
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    if union is None:
        union = (torch.empty((B, h_kv, group * k), dtype=torch.int32, device=dev),
                 torch.empty((B, h_kv, group * k), dtype=torch.uint8, device=dev),
                 torch.empty((B, h_kv), dtype=torch.int32, device=dev))
    if workspace is None:
        n = union_workspace_size(B, h_kv, group, d, cache.page_size, cache.dtype, k)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    ul, um, uc = union
    _check(lib().quest_union_decode_attn(
        ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q), int(group), _ptr(sel_logical),
        int(k), _ptr(out), _ptr(lse), float(sm_scale), _ptr(ul), _ptr(um), _ptr(uc),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream(stream)))
    return out, lse, union


def select_topk(table: PageTable, h_kv: int, page_size: int, scores, k: int,
                out=None, stream=None, n_sink: int = 0, n_local: int = 0):
    """quest_select_topk: (sel_logical, sel_phys [B, h_kv, k], sel_count [B, h_kv]).
    n_sink / n_local: first / last valid pages always kept (hybrid budget)."""
    if out is None:
        dev = scores.device
        out = (torch.empty((table.batch, h_kv, k), dtype=torch.int32, device=dev),
               torch.empty((table.batch, h_kv, k), dtype=torch.int32, device=dev),
               torch.empty((table.batch, h_kv), dtype=torch.int32, device=dev))
    sl, sp, sc = out
    _check(lib().quest_select_topk(ctypes.byref(table.c), int(h_kv), int(page_size),
                                   _ptr(scores), int(k), int(n_sink), int(n_local),
                                   _ptr(sl), _ptr(sp), _ptr(sc), _stream(stream)))
    return sl, sp, sc


def attn_workspace_size(batch, h_kv, group, head_dim, page_size, k) -> int:
    return int(lib().quest_attn_workspace_size(batch, h_kv, group, head_dim, page_size, k))


def sparse_decode_attn(cache: PagedCache, table: PageTable, q, group: int, sel_logical,
                       sel_phys, k: int, out=None, lse=None, sm_scale: float = 0.0,
                       workspace=None, stream=None):
    """quest_sparse_decode_attn: (out [B, h_q, d] fp32, lse [B, h_q] fp32)."""
    B, h_q, d = q.shape
    dev = q.device
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    if workspace is None:
        n = attn_workspace_size(B, cache.h_kv, group, d, cache.page_size, k)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    _check(lib().quest_sparse_decode_attn(
        ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q), int(group), _ptr(sel_logical),
        _ptr(sel_phys), int(k), _ptr(out), _ptr(lse), float(sm_scale), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream(stream)))
    return out, lse


def diag_workspace_size(h_kv, group, nnz, page_size) -> int:
    return int(lib().quest_diag_workspace_size(h_kv, group, nnz, page_size))


def recall_diagnostics(cache: PagedCache, table: PageTable, q, group: int, sel_logical,
                       k: int, top_r: int, sm_scale: float = 0.0, workspace=None, stream=None):
    """quest_recall_diagnostics: dict of slack [h_q, nnz], eps [B, h_q],
    topr [B, h_q] and vmax [B, h_kv] (fp32)."""
    B, h_q, d = q.shape
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(slack=torch.empty((h_q, table.nnz), **f32), eps=torch.empty((B, h_q), **f32),
               topr=torch.empty((B, h_q), **f32), vmax=torch.empty((B, cache.h_kv), **f32))
    if workspace is None:
        n = diag_workspace_size(cache.h_kv, group, table.nnz, cache.page_size)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    _check(lib().quest_recall_diagnostics(
        ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q), int(group), _ptr(sel_logical),
        int(k), int(top_r), float(sm_scale), _ptr(out["slack"]), _ptr(out["eps"]),
        _ptr(out["topr"]), _ptr(out["vmax"]), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream(stream)))
    return out


def decode_workspace_size(batch, nnz, h_kv, group, head_dim, page_size, dtype, k) -> int:
    return int(lib().quest_decode_workspace_size(batch, nnz, h_kv, group, head_dim, page_size,
                                                 dtype_code(dtype), k))


class DecodeStep:
    """Buffers of quest_decode_step for a fixed problem shape: scores,
    selections, outputs and a zero-filled workspace (reused across calls).
    n_sink / n_local: first / last valid pages always kept (hybrid budget)."""

    def __init__(self, cache: PagedCache, table: PageTable, group: int, k: int, device=None,
                 n_sink: int = 0, n_local: int = 0):
        dev = device or cache.k_pool.device
        B, h = table.batch, cache.h_kv
        self.group, self.k = group, k
        self.n_sink, self.n_local = n_sink, n_local
        self.scores = torch.empty((h, max(table.nnz, 1)), dtype=torch.float32, device=dev)
        self.sel = (torch.empty((B, h, k), dtype=torch.int32, device=dev),
                    torch.empty((B, h, k), dtype=torch.int32, device=dev),
                    torch.empty((B, h), dtype=torch.int32, device=dev))
        self.out = torch.empty((B, h * group, cache.head_dim), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, h * group), dtype=torch.float32, device=dev)
        n = decode_workspace_size(B, table.nnz, h, group, cache.head_dim, cache.page_size,
                                  cache.dtype, k)
        if n == 0:
            raise RuntimeError("quest_decode_step does not support this shape")
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=dev)

    def __call__(self, cache: PagedCache, table: PageTable, q, k_new=None, v_new=None,
                 sm_scale: float = 0.0, stream=None):
        sl, sp, sc = self.sel
        _check(lib().quest_decode_step(
            ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(k_new), _ptr(v_new), _ptr(q),
            int(self.group), int(self.k), int(self.n_sink), int(self.n_local),
            _ptr(self.scores), _ptr(sl), _ptr(sp), _ptr(sc),
            _ptr(self.out), _ptr(self.lse), float(sm_scale), _ptr(self.workspace),
            int(self.workspace.numel()), _stream(stream)))
        return self.out, self.lse


def decode_step_kernel(batch, h_kv, group, head_dim, page_size, dtype, k, summary_fp8=False) -> str:
    """quest_decode_step_kernel: the kernel quest_decode_step launches for
    these sizes on the current device ("cstep_kernel", "step_kernel", or ""
    if unsupported)."""
    r = int(lib().quest_decode_step_kernel(int(batch), int(h_kv), int(group), int(head_dim),
                                           int(page_size), dtype_code(dtype), int(k),
                                           int(bool(summary_fp8))))
    return {2: "cstep_kernel", 1: "step_kernel"}.get(r, "")


TRACE_NAMES = ("start", "scored", "selected", "att_start", "att_pages", "att_merged",
               "sel_begin", "sel_end", "", "exit",
               "sel0_polled | desc0", "sel0_done | page0", "sel1_polled | merged",
               "sel1_done | fmerge0", "sel2_polled | fmerge1", "sel2_done")
# slots 6-7: the first select's start (after the scored gate) and the last
# select's end, on every CTA that selects; slots 10-15 depend on the CTA's
# role: select stamps on dedicated selectors (the CTAs whose "scored" stamp
# precedes any scoring), attention and final-merge stamps on the others

# the cluster kernel's slots (unused ones empty)
CTRACE_NAMES = ("start", "prev_waited", "", "", "att_tile0", "keys_in", "sel_published",
                "merged_last", "", "exit", "topk_done", "phys_done", "", "", "", "")


def set_trace(buffer, max_ctas=0, batch=0, h_kv=0, group=1, head_dim=128, page_size=16,
              dtype=torch.float16, k=1) -> int:
    """quest_set_trace: per-CTA phase stamps of later decode steps into
    `buffer` (uint64 device tensor of 16 * max_ctas entries); None disables.
    Returns the grid size used for the given shape."""
    return int(lib().quest_set_trace(_ptr(buffer), int(max_ctas), int(batch), int(h_kv),
                                     int(group), int(head_dim), int(page_size),
                                     dtype_code(dtype), int(k)))


def sparse_decode_attn_noalloc(cache: PagedCache, table: PageTable, q, group: int,
                               sel_logical, sel_phys, k: int, out=None, lse=None,
                               sm_scale: float = 0.0, stream=None):
    """quest_sparse_decode_attn_noalloc: the same attention with the split-K
    partials in the library's fixed 4 MiB buffer (for callers that cannot
    allocate device memory); calls on overlapping streams race on it."""
    B, h_q, d = q.shape
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=q.device)
    _check(lib().quest_sparse_decode_attn_noalloc(
        ctypes.byref(cache.c), ctypes.byref(table.c), _ptr(q), int(group), _ptr(sel_logical),
        _ptr(sel_phys), int(k), _ptr(out), _ptr(lse), float(sm_scale), _stream(stream)))
    return out, lse


def test_step_fault(mode: int, wait_limit: int = 0) -> None:
    """quest_test_step_fault: mode 1 makes a wait of later decode steps on the
    cluster kernel run out, mode 2 one of later attention calls; under
    `wait_limit` tries per wait (0 = default). Mode 0 restores normal
    operation."""
    _check(lib().quest_test_step_fault(int(mode), int(wait_limit)))


def device_error(stream=None) -> int:
    """Synchronise and return (then clear) the device error word."""
    v = int(lib().quest_get_device_error(_stream(stream)))
    if v < 0:
        raise RuntimeError("quest_get_device_error: CUDA call failed")
    return v
