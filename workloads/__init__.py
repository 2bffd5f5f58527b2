"""Seeded synthetic inputs shaped like the Quest page's decode workloads.

This module only *makes inputs*: page tables, token K/V, queries and the
placement of tokens into a paged pool. It holds none of the method's
arithmetic (no summaries, bounds, selection or attention), so both the CUDA
path and the fp64 oracle can take their inputs from it.

Every tensor is drawn from a ``torch.Generator`` seeded from the workload's
seed, on the device the caller asks for; the GPU path and the oracle always
consume the *same stored tensors* (the oracle gets host copies), so no
cross-device bit agreement of the generator is needed.

Workloads (Llama-2-7B-like MHA shapes of the Quest page's intro and §2):

``tiny``          1 request, 1 KV head, d=64, S=16, 1000 tokens (63 pages,
                  8 valid in the tail), K=8, fp32 N(0,1).
``llama_layer``   1 request, 32 heads (MHA), d=128, S=16, 32768 tokens,
                  budget 2048 tokens (K=128), fp16 N(0,1) keys with 4 outlier
                  channels x8, rotate-half RoPE (base 10000) on K and q.
``llama_step``    ``llama_layer`` x 32 layers; layers 0-1 dense, 2-31 Quest
                  with budgets 1024 / 2048 / 4096 tokens.
``gqa_batch``     16 requests, lengths U[8192, 131072], 8 KV heads x 4 query
                  heads, d=128, S=16, K=256, random physical page permutation.
``append_128k``   1 request, 32 heads, d=128, S=32, prefill 131072 tokens then
                  64 single-token decode steps, budget 4096 tokens (K=128).
``gqa_small``     ``gqa_batch``'s shapes with 4 requests of U[16384, 32768]
                  tokens (a small case for profiler captures).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_kv: int
    group: int
    head_dim: int
    page_size: int
    k: int                      # pages selected per (request, KV head)
    dtype: torch.dtype
    seed: int
    seq_lens: tuple = ()        # fixed lengths; empty => drawn from len_range
    len_range: tuple = ()       # inclusive [lo, hi] for seeded lengths
    rope: bool = False
    outlier_channels: int = 0
    outlier_scale: float = 8.0
    permute_pages: bool = False
    layers: int = 1
    dense_layers: int = 0
    budgets: tuple = ()         # token budgets swept (llama_step)
    decode_steps: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def h_q(self) -> int:
        return self.h_kv * self.group

    def lengths(self) -> np.ndarray:
        if self.seq_lens:
            return np.asarray(self.seq_lens, dtype=np.int64)
        g = torch.Generator().manual_seed(self.seed * 7919 + 17)
        lo, hi = self.len_range
        return torch.randint(lo, hi + 1, (self.batch,), generator=g).numpy().astype(np.int64)


WORKLOADS = {
    "tiny": Workload("tiny", batch=1, h_kv=1, group=1, head_dim=64, page_size=16,
                     k=8, dtype=torch.float32, seed=1001, seq_lens=(1000,)),
    "llama_layer": Workload("llama_layer", batch=1, h_kv=32, group=1, head_dim=128,
                            page_size=16, k=128, dtype=torch.float16, seed=1002,
                            seq_lens=(32768,), rope=True, outlier_channels=4),
    "llama_step": Workload("llama_step", batch=1, h_kv=32, group=1, head_dim=128,
                           page_size=16, k=128, dtype=torch.float16, seed=1003,
                           seq_lens=(32768,), rope=True, outlier_channels=4,
                           layers=32, dense_layers=2, budgets=(1024, 2048, 4096)),
    "gqa_batch": Workload("gqa_batch", batch=16, h_kv=8, group=4, head_dim=128,
                          page_size=16, k=256, dtype=torch.float16, seed=1004,
                          len_range=(8192, 131072), permute_pages=True),
    "append_128k": Workload("append_128k", batch=1, h_kv=32, group=1, head_dim=128,
                            page_size=32, k=128, dtype=torch.float16, seed=1005,
                            seq_lens=(131072,), decode_steps=64),
    # gqa_batch's shapes at a quarter of its requests and lengths (about 0.4 GB of
    # K/V, still above the 129 MB L2): the small case the profiler captures
    "gqa_small": Workload("gqa_small", batch=4, h_kv=8, group=4, head_dim=128,
                          page_size=16, k=256, dtype=torch.float16, seed=1006,
                          len_range=(16384, 32768), permute_pages=True),
}


# ---------------------------------------------------------------------------
# Page tables
# ---------------------------------------------------------------------------

@dataclass
class PageTable:
    page_indptr: np.ndarray     # int32 [batch+1]
    page_indices: np.ndarray    # int32 [nnz]
    seq_lens: np.ndarray        # int32 [batch]
    n_phys: int
    page_size: int

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    @property
    def nnz(self) -> int:
        return int(self.page_indptr[-1])

    def pages_of(self, r: int) -> int:
        return int(self.page_indptr[r + 1] - self.page_indptr[r])


def make_page_table(seq_lens, page_size, *, seed=0, permute=False,
                    spare_pages=0, reserve_tokens=0) -> PageTable:
    """CSR page table for the given lengths.

    Each request gets ceil((len + reserve_tokens) / S) logical pages. Physical
    pages are 0..nnz-1 in request order, or a seeded random permutation of a
    pool with ``spare_pages`` unused extra pages when ``permute`` is set.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    counts = (seq_lens + reserve_tokens + page_size - 1) // page_size
    indptr = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(counts)
    nnz = int(indptr[-1])
    n_phys = nnz + spare_pages
    if permute:
        g = torch.Generator().manual_seed(seed * 104729 + 3)
        perm = torch.randperm(n_phys, generator=g).numpy()[:nnz]
    else:
        perm = np.arange(nnz)
    return PageTable(indptr.astype(np.int32), perm.astype(np.int32),
                     seq_lens.astype(np.int32), n_phys, page_size)


# ---------------------------------------------------------------------------
# Token K/V and queries
# ---------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """Seeded N(0,1) drawn in fp32 and rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    return x.to(dtype)


def rope_rotate(x: torch.Tensor, positions: torch.Tensor, base=10000.0) -> torch.Tensor:
    """Rotate-half RoPE in fp64: pairs (j, j + d/2), theta_i = base^(-2i/d).

    x is [n, heads, d]; positions is [n]. Returns fp64. (Input preparation:
    the cache holds post-RoPE keys, as the Quest page §1.1 requires of the
    summary's coordinates.)
    """
    d = x.shape[-1]
    half = d // 2
    xd = x.to(torch.float64)
    i = torch.arange(half, device=x.device, dtype=torch.float64)
    inv = base ** (-2.0 * i / d)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]       # [n, half]
    cos = torch.cos(ang)[:, None, :]
    sin = torch.sin(ang)[:, None, :]
    x1, x2 = xd[..., :half], xd[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def layer_seed(w: Workload, layer: int) -> int:
    return w.seed * 1000 + layer


def outlier_channels(w: Workload, layer: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(layer_seed(w, layer) + 11)
    return torch.randperm(w.head_dim, generator=g)[: w.outlier_channels]


def request_tokens(w: Workload, r: int, length: int, layer=0, device="cpu",
                   start=0):
    """K and V for tokens start..start+length-1 of request r: [length, h_kv, d].

    Token t of request r is drawn from a stream keyed by (seed, layer, r), so a
    prefix generated alone equals the same prefix of a longer draw only when
    ``start`` is 0; decode tokens use their own stream via ``start``.
    """
    s = layer_seed(w, layer) * 131 + r * 7 + (start * 1000003)
    k = normal((length, w.h_kv, w.head_dim), s + 1, device)
    v = normal((length, w.h_kv, w.head_dim), s + 2, device)
    if w.outlier_channels:
        ch = outlier_channels(w, layer).to(k.device)
        k[..., ch] *= w.outlier_scale
    if w.rope:
        pos = torch.arange(start, start + length, device=k.device)
        k = rope_rotate(k, pos)
    return k.to(w.dtype), v.to(w.dtype)


def queries(w: Workload, positions, layer=0, device="cpu", step=0) -> torch.Tensor:
    """Decode queries [batch, h_q, d]; with RoPE, request r's query sits at
    positions[r] (the position of the token being decoded)."""
    s = layer_seed(w, layer) * 131 + 5 + step * 7777
    q = normal((w.batch, w.h_q, w.head_dim), s, device)
    if w.rope:
        pos = torch.as_tensor(np.asarray(positions), device=q.device)
        q = rope_rotate(q, pos)
    return q.to(w.dtype)


def tokens_for_table(w: Workload, table: PageTable, layer=0, device="cpu"):
    """Concatenated K/V of all requests in request order, plus the CSR
    ``append_indptr`` [batch+1] over them."""
    ks, vs = [], []
    indptr = [0]
    for r in range(table.batch):
        L = int(table.seq_lens[r])
        k, v = request_tokens(w, r, L, layer, device)
        ks.append(k)
        vs.append(v)
        indptr.append(indptr[-1] + L)
    return (torch.cat(ks), torch.cat(vs), np.asarray(indptr, dtype=np.int32))


def empty_pool(table: PageTable, h_kv, d, dtype, device="cpu", poison=True):
    """Pool tensors [n_phys, h_kv, S, d] and summary [n_phys, h_kv, 2, d].

    With ``poison`` the never-written slots hold NaN so that any read of an
    invalid slot shows up in the results.
    """
    fill = float("nan") if poison else 0.0
    shape = (table.n_phys, h_kv, table.page_size, d)
    k_pool = torch.full(shape, fill, dtype=dtype, device=device)
    v_pool = torch.full(shape, fill, dtype=dtype, device=device)
    summ = torch.full((table.n_phys, h_kv, 2, d), fill, dtype=dtype, device=device)
    return k_pool, v_pool, summ


def place_tokens(pool: torch.Tensor, table: PageTable, tokens: torch.Tensor,
                 append_indptr, seq_lens_before=None):
    """Copy token rows into their (page, slot) places: pure data placement.

    Token i of request r goes to position seq_lens_before[r] + (i - start_r).
    """
    S = table.page_size
    dev = pool.device
    rows, phys, slots = [], [], []
    for r in range(table.batch):
        a, b = int(append_indptr[r]), int(append_indptr[r + 1])
        if b == a:
            continue
        base = 0 if seq_lens_before is None else int(seq_lens_before[r])
        pos = np.arange(base, base + (b - a))
        lp = pos // S
        phys.append(table.page_indices[table.page_indptr[r] + lp])
        slots.append(pos % S)
        rows.append(np.arange(a, b))
    if not rows:
        return pool
    rows = torch.as_tensor(np.concatenate(rows), device=dev)
    phys = torch.as_tensor(np.concatenate(phys).astype(np.int64), device=dev)
    slots = torch.as_tensor(np.concatenate(slots), device=dev)
    pool[phys, :, slots, :] = tokens[rows].to(pool.dtype)
    return pool


def selection_budget(budget_tokens: int, page_size: int) -> int:
    """Pages selected for a token budget B = K * S (Quest page §2)."""
    return budget_tokens // page_size


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
