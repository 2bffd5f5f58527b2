#!/usr/bin/env python
"""Decode-step benchmark of the Quest hot path on one GB300.

One step = one decode step of one attention layer for the Llama-2-7B-shaped
workload (1 request, 32 heads, d_h 128, 32768-token context, page size 16,
token budget 2048 -> K = 128 pages, fp16): append the new token's K/V (and
its page summary), score all 2048 pages, select the top 128 per head, attend
over the selected pages (split-K + combine). Steps run as CUDA-graph replays.

Output: one JSON line (rank 0). `value` is the device-timed latency per layer
(µs, lower is better) with inputs resident in HBM; `e2e` is the same step
with the per-step inputs (q, new k/v) copied from pinned host memory and the
output read back, host wall clock per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")          # the CPU oracle runs on one core

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "sparse decode-attn latency (µs/layer) & achieved HBM GB/s vs roofline"
UNIT = "us/layer"
MIB = 1 << 20


# ---------------------------------------------------------------------------
# Byte accounting (Quest page §2 eq (9)-(12)): algorithmic bytes of one step
# ---------------------------------------------------------------------------

def step_bytes(n_pages, h_kv, group, d, S, k_sel_pages, valid_tokens_selected, esize,
               append_tokens=1, batch=1, kv_tokens_total=None, summary_esize=None):
    """Algorithmic bytes of one decode step of one layer.

    summary of every scored page (index term, eq (10)) + K/V of the valid
    tokens of the selected pages (eq (11)) + q read + o written (fp32) + the
    append (new k/v read, written to the pool, tail-page summary read+write).
    Scores, ids and split-K partials are intermediates and not counted.
    n_pages: scored pages of all requests; valid_tokens_selected: per (request,
    KV head) when all are alike, else kv_tokens_total sums them over both.
    summary_esize: bytes per summary element (1 for E4M3 codes; default esize).
    """
    sz = esize if summary_esize is None else summary_esize
    summary = n_pages * h_kv * 2 * d * sz
    kv_tok = valid_tokens_selected * h_kv if kv_tokens_total is None else kv_tokens_total
    kv = kv_tok * 2 * d * esize
    q = batch * h_kv * group * d * esize
    o = batch * h_kv * group * d * 4
    append = batch * (append_tokens * h_kv * d * esize * 2 * 2 + h_kv * 2 * d * sz * 2)
    return dict(summary=summary, kv=kv, q=q, o=o, append=append,
                total=summary + kv + q + o + append)


def paper_traffic_ratio(L, S, budget_tokens):
    """rho = 1/S + K/P (eq (12)) for a token budget B = K*S."""
    K = budget_tokens // S
    return 1.0 / S + K / (L / S)


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v
                          and "Not" not in v})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].strip() not in ("", "[N/A]"))}


def workload_config(w: wl.Workload):
    """The bench line's `config`: the workload by what it is, with its sizes."""
    lens = w.lengths().astype(np.int64)
    B = len(lens)
    heads = (f"{w.h_kv} heads (MHA)" if w.group == 1
             else f"{w.h_kv} KV heads x {w.group} query heads (GQA, group max)")
    ctx = (f"context {int(lens[0])}" if B == 1 else
           f"contexts {int(lens.min())}-{int(lens.max())} (total {int(lens.sum())})")
    dt = "fp16" if w.dtype == torch.float16 else "fp32"
    desc = (f"{w.name}: {B} request{'s' if B > 1 else ''}, {heads}, d_h {w.head_dim}, {ctx}, "
            f"page {w.page_size}, budget {w.k * w.page_size} tokens (K={w.k}), {dt}"
            + (", RoPE" if w.rope else "") + (", physical pages permuted" if w.permute_pages else "")
            + (f", {w.layers} layers (first {w.dense_layers} dense, K = P), budget sweep "
               f"{'/'.join(str(b) for b in w.budgets)} tokens" if w.layers > 1 else ""))
    cfg = {"workload": desc, "n_pages": int((-(-lens // w.page_size)).sum()), "k": w.k,
           "h_kv": w.h_kv, "group": w.group, "head_dim": w.head_dim,
           "page_size": w.page_size, "seq_len": int(lens[0]) if B == 1 else int(lens.sum())}
    if B > 1:
        cfg["batch"] = B
    return cfg


def data_desc(w: wl.Workload):
    """The bench line's `data`: how the synthetic inputs are made."""
    extra = ""
    if w.outlier_channels:
        extra += f", {w.outlier_channels} outlier channels x{w.outlier_scale:g}"
    if w.rope:
        extra += ", RoPE"
    return f"synthetic (seeded N(0,1) K/V/q{extra})"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# Workload set-up on the device
# ---------------------------------------------------------------------------

class LayerSetup:
    """One attention layer of the workload: pools built by the library's own
    append (prefill of all but the last token of each request), plus each
    request's decode token and query."""

    def __init__(self, w: wl.Workload, nbuf: int, dev, sample_heads=4, n_sink=0, n_local=0,
                 summary_fp8=False, prefill_reps=5):
        import query_aware_sparse_gb300 as qs
        self.qs = qs
        self.w = w
        self.summary_fp8 = summary_fp8
        lens = w.lengths().astype(np.int64)
        B = len(lens)
        self.lens, self.L = lens, int(lens[0])
        S, h, d = w.page_size, w.h_kv, w.head_dim
        t = wl.make_page_table(lens, S, seed=w.seed, permute=w.permute_pages,
                               spare_pages=64 if w.permute_pages else 0)
        self.table_np = t
        k_tok, v_tok, ind = wl.tokens_for_table(w, t, device=dev)
        self.q = wl.queries(w, lens - 1, device=dev)
        # host copies of request 0's inputs (every head), for the oracle
        L0 = int(lens[0])
        self.sample = (k_tok[:L0].cpu(), v_tok[:L0].cpu(), self.q[:1].cpu())
        i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32), device=dev)
        self.table = qs.PageTable(i32(t.page_indptr), i32(t.page_indices), i32(lens))
        kp, vp, sm = wl.empty_pool(t, h, d, w.dtype, device=dev, poison=False)
        if summary_fp8:            # E4M3 codes with directed rounding instead
            sm = torch.zeros(sm.shape, dtype=torch.uint8, device=dev)
        self.caches = [qs.PagedCache(kp, vp, sm)]
        # prefill append of all but the last token of each request through
        # the library (timed once)
        pre = qs.PageTable(self.table.page_indptr, self.table.page_indices, i32(lens - 1))
        rows = torch.cat([torch.arange(int(ind[r]), int(ind[r]) + int(lens[r]) - 1, device=dev)
                          for r in range(B)])
        kpre, vpre = k_tok[rows].contiguous(), v_tok[rows].contiguous()
        pre_ind = np.concatenate([[0], np.cumsum(lens - 1)])
        torch.cuda.synchronize()
        # the first call, then repeats (each page starts over from its slot 0,
        # so a repeat rewrites the same pool and summaries): the median of the
        # repeats is the prefill's time, the first call is reported beside it
        ind_d, zero_d = i32(pre_ind), i32(np.zeros(B))
        pre_ms = []
        for _ in range(1 + prefill_reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            qs.append_kv(self.caches[0], pre, kpre, vpre, ind_d, zero_d)
            e1.record()
            torch.cuda.synchronize()
            pre_ms.append(e0.elapsed_time(e1))
        n_pre = int(pre_ind[-1])
        # read K and V rows, write them into the pool, write every page's summary
        pre_bytes = (n_pre * h * d * k_tok.element_size() * 4 +
                     int(-(-(lens - 1) // S).sum()) * h * 2 * d * sm.element_size())
        med = statistics.median(pre_ms[1:]) if prefill_reps else pre_ms[0]
        self.prefill = {"tokens": n_pre, "bytes": pre_bytes, "ms": med, "GBps": pre_bytes / med / 1e6,
                        "first_call_ms": pre_ms[0], "reps": prefill_reps}
        assert qs.device_error() == 0
        for _ in range(nbuf - 1):   # distinct copies: each step reads cold memory
            c = self.caches[0]
            self.caches.append(qs.PagedCache(c.k_pool.clone(), c.v_pool.clone(), c.summary.clone()))
        last = torch.as_tensor(ind[:-1] + lens - 1, device=dev)
        self.k_dec = k_tok[last].contiguous()
        self.v_dec = v_tok[last].contiguous()
        del k_tok, v_tok, kpre, vpre
        torch.cuda.empty_cache()
        self.app_indptr = i32(np.arange(B + 1))
        self.before = i32(lens - 1)
        self.K = w.k
        hq = h * w.group
        self.scores = torch.empty((h, t.nnz), dtype=torch.float32, device=dev)
        self.sel = (torch.empty((B, h, self.K), dtype=torch.int32, device=dev),
                    torch.empty((B, h, self.K), dtype=torch.int32, device=dev),
                    torch.empty((B, h), dtype=torch.int32, device=dev))
        self.out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
        n = qs.attn_workspace_size(B, h, w.group, d, S, self.K)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev)
        self.n_sink, self.n_local = n_sink, n_local
        self.fused = qs.DecodeStep(self.caches[0], self.table, w.group, self.K,
                                   n_sink=n_sink, n_local=n_local)
        self.out, self.lse = self.fused.out, self.fused.lse

    # the four stages of one decode step on cache copy b
    def append(self, b):
        self.qs.append_kv(self.caches[b], self.table, self.k_dec, self.v_dec,
                          self.app_indptr, self.before)

    def score(self, b):
        self.qs.score_pages(self.caches[b], self.table, self.q, self.w.group, self.scores)

    def select(self, b):
        self.qs.select_topk(self.table, self.w.h_kv, self.w.page_size, self.scores, self.K,
                            out=self.sel, n_sink=self.n_sink, n_local=self.n_local)

    def attend(self, b):
        self.qs.sparse_decode_attn(self.caches[b], self.table, self.q, self.w.group,
                                   self.sel[0], self.sel[1], self.K, self.out, self.lse,
                                   workspace=self.ws)

    def unfused(self, b):
        self.append(b)
        self.score(b)
        self.select(b)
        self.attend(b)

    def step(self, b):
        """The fused decode step: append + score + select + attention in one launch."""
        self.fused(self.caches[b], self.table, self.q, self.k_dec, self.v_dec)

    KERNELS_PER_STEP = 1   # quest_decode_step is one kernel launch

    def bytes(self):  # noqa: A003
        """Algorithmic bytes of one step: the summaries of every valid page and
        the K/V of the valid tokens of the pages the last fused step chose."""
        w, S = self.w, self.w.page_size
        P = -(-self.lens // S)
        sl = self.fused.sel[0].cpu().numpy()                 # [B, h_kv, K] logical ids
        lens = self.lens[:, None, None]
        valid = np.where(sl >= 0, np.clip(lens - sl.astype(np.int64) * S, 0, S), 0)
        return step_bytes(int(P.sum()), w.h_kv, w.group, w.head_dim, S, self.K, 0,
                          self.k_dec.element_size(), batch=len(self.lens),
                          kv_tokens_total=int(valid.sum()),
                          summary_esize=self.caches[0].summary.element_size())


def time_stage(fn, nbuf, reps):
    """Average device time (ms) of one call of fn(b): a CUDA graph holds one
    call per cache copy back to back; it is replayed `reps` times between two
    events on the capturing stream, so host launch cost is not included."""
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for b in range(nbuf):
                fn(b)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * nbuf)


def source_hash(*names):
    """Hash of the kernel sources as compiled: comments and blank space do
    not count (an edit to a comment leaves recorded counters valid)."""
    import re
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "query_aware_sparse_gb300", "csrc", n)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, workload):
    """dram bytes per launch recorded from an ncu capture, if the kernel's
    source is unchanged since; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    e = rec.get(f"{kernel_key}@{workload}")      # one record per kernel and workload
    if not e:
        return None
    try:
        if e.get("source_hash") != source_hash(*e["sources"]):
            return None
    except OSError:                  # a recorded source no longer exists
        return None
    return e["dram_bytes_per_launch"]


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------

class OracleSample:
    """The oracle's decode step on a sample of the heads of the same layer,
    built from the generated inputs (never from the device path's results)."""

    def __init__(self, w: wl.Workload, k_tok, v_tok, q, heads: int, n_sink=0, n_local=0,
                 summary_fp8=False, k=None):
        from oracle import quest_oracle as qo
        self.qo = qo
        self.summary_fp8 = summary_fp8
        self.n_sink, self.n_local = n_sink, n_local
        self.heads = heads
        self.w = w
        self.k = w.k if k is None else k          # pages selected (K = P: dense)
        L = int(w.lengths()[0])
        self.L = L
        t = wl.make_page_table([L], w.page_size, seed=w.seed)
        self.t = t
        k_tok, v_tok = k_tok[:, :heads], v_tok[:, :heads]
        kp, vp, _ = wl.empty_pool(t, heads, w.head_dim, w.dtype, poison=True)
        ind = np.array([0, L - 1])
        wl.place_tokens(kp, t, k_tok[:L - 1], ind)
        wl.place_tokens(vp, t, v_tok[:L - 1], ind)
        self.kp, self.vp = kp.numpy(), vp.numpy()
        self.q = q[:, :heads * w.group].numpy()
        self.kdec = k_tok[L - 1:L].numpy()
        self.vdec = v_tok[L - 1:L].numpy()
        self.sm = qo.build_summary(self.kp, t.page_indptr, t.page_indices,
                                   np.array([L - 1], np.int32))

    def step(self):
        qo, t, w = self.qo, self.t, self.w
        qo.append_kv(self.kp, self.vp, self.sm, t.page_indptr, t.page_indices,
                     np.array([self.L - 1]), np.array([0, 1]), self.kdec, self.vdec)
        if self.summary_fp8:      # the oracle rounds its exact summary out to E4M3
            codes, _ = qo.summary_to_e4m3(self.sm)
            sc = qo.score_pages_e4m3(self.q, codes, t.page_indptr, t.page_indices, w.group)
        else:
            sc = qo.score_pages(self.q, self.sm, t.page_indptr, t.page_indices, w.group)
        sel, _, _ = qo.select_hybrid(sc, t.page_indptr, t.page_indices, np.array([self.L]),
                                     w.page_size, self.k, self.n_sink, self.n_local)
        qo.sparse_attention(self.q, self.kp, self.vp, t.page_indptr, t.page_indices,
                            np.array([self.L], np.int32), sel, w.group)

    def time_steps(self, n):
        ts = []
        for _ in range(n):
            t0 = time.perf_counter()
            self.step()
            ts.append(time.perf_counter() - t0)
        # µs per full layer: all KV heads, all requests (by their pages)
        return [x * 1e6 * self.w.h_kv / self.heads * pages_scale(self.w) for x in ts]


def pages_scale(w: wl.Workload) -> float:
    """All requests' pages over request 0's: the oracle samples request 0."""
    lens = w.lengths().astype(np.int64)
    pages = -(-lens // w.page_size)
    return float(pages.sum()) / float(pages[0])


def _oracle_proc(conn, barrier):
    """A worker of OraclePool (a spawned process on one core): builds oracle
    samples when asked, and times rounds over them, starting together with
    the other workers at a barrier."""
    torch.set_num_threads(1)
    samples = []
    while True:
        msg = conn.recv()
        if msg[0] == "build":
            samples.append(OracleSample(*msg[1], **msg[2]))
            conn.send(None)
        elif msg[0] == "clear":
            samples = []
            conn.send(None)
        elif msg[0] == "time":
            for o in samples:                       # warm
                o.step()
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            for _ in range(msg[1]):
                for o in samples:
                    o.step()
            conn.send((t0, time.perf_counter()))
        else:
            return


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """The oracle on several host cores at once: one spawned single-threaded
    process per core, each over its own (layer, KV head) units of request 0
    (independent work), timed from a common start to the last finish."""

    def __init__(self, n: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n = n
        self.barrier = ctx.Barrier(n)
        self.conns, self.procs = [], []
        for _ in range(n):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_proc, args=(b, self.barrier), daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)

    def build(self, w, k_tok, v_tok, q, k=None, n_sink=0, n_local=0, summary_fp8=False):
        """Worker i takes KV heads [i h_kv / n, (i + 1) h_kv / n) of these
        inputs (request 0, one layer; all heads)."""
        h, G = w.h_kv, w.group
        for c in self.conns:
            c.send(("clear",))
            c.recv()
        for i, c in enumerate(self.conns):
            h0, h1 = i * h // self.n, (i + 1) * h // self.n
            c.send(("build", (w, k_tok[:, h0:h1].contiguous(), v_tok[:, h0:h1].contiguous(),
                              q[:, h0 * G:h1 * G].contiguous(), h1 - h0, n_sink, n_local),
                    {"summary_fp8": summary_fp8, "k": k}))
        for c in self.conns:
            c.recv()

    def time(self, rounds: int) -> float:
        """Seconds per round of every worker's units."""
        for c in self.conns:
            c.send(("time", rounds))
        res = [c.recv() for c in self.conns]
        return (max(r[1] for r in res) - min(r[0] for r in res)) / rounds

    def close(self):
        for c in self.conns:
            c.send(("stop",))
        for p in self.procs:
            p.join(timeout=30)


# ---------------------------------------------------------------------------
# Main
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks of the process group (the job ends with
    its slowest replica); x itself without a group or with one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama_layer")
    ap.add_argument("--nbuf", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-heads", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="oracle timing budget for cpu_baseline (0 = skip)")
    ap.add_argument("--stage-reps", type=int, default=100)
    ap.add_argument("--sink-tokens", type=int, default=0,
                    help="hybrid budget: sink tokens kept (whole pages, ceil)")
    ap.add_argument("--local-tokens", type=int, default=0,
                    help="hybrid budget: recent-window tokens kept (whole pages, ceil)")
    ap.add_argument("--diagnostics", type=int, default=0, metavar="R",
                    help="also time quest_recall_diagnostics with top-R = R (0 = off)")
    ap.add_argument("--gqa-union", action="store_true",
                    help="also time GQA per-query-head selection with the per-KV-head page union")
    ap.add_argument("--summary", choices=["kv", "e4m3"], default="kv",
                    help="page summaries in the K/V dtype or as E4M3 codes (directed rounding)")
    args = ap.parse_args(argv)
    assert args.warmup >= 3, "at least 3 warm-up steps"

    ws, rank, local = dist_env()
    if args.impl == "reference" and rank != 0:
        return          # the oracle arm runs on rank 0 alone; other ranks do no work
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1 and args.impl != "reference":   # the oracle arm needs no group
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = wl.WORKLOADS[args.workload]
    cfg = workload_config(w)

    n_sink = -(-args.sink_tokens // w.page_size)
    n_local = -(-args.local_tokens // w.page_size)
    if n_sink or n_local:
        # Quest page 2.2: the budget keeps its page count; sinks and the window
        # take whole pages out of it and Quest gets the rest
        cfg["hybrid"] = {"sink_tokens": args.sink_tokens, "local_tokens": args.local_tokens,
                         "sink_pages": n_sink, "local_pages": n_local,
                         "quest_pages": w.k - n_sink - n_local}
    args.n_sink, args.n_local = n_sink, n_local
    args.summary_fp8 = args.summary == "e4m3"
    if args.summary_fp8:
        cfg["summary_dtype"] = "e4m3 (min toward -inf, max toward +inf)"

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, w, cfg, dev, ws)
        return

    import query_aware_sparse_gb300 as qs
    qs.lib()
    if w.layers > 1:
        run_model_step(args, w, cfg, dev, ws, rank, local)
        return
    setup = LayerSetup(w, args.nbuf, dev, sample_heads=args.cpu_heads,
                       n_sink=n_sink, n_local=n_local, summary_fp8=args.summary_fp8)
    cfg["l2"] = (f"rotating {args.nbuf} distinct copies of the layer "
                 f"({args.nbuf * (setup.caches[0].k_pool.nbytes * 2 + setup.caches[0].summary.nbytes) / 2**30:.1f} GiB)"
                 " so every step reads memory not touched in the previous "
                 f"{args.nbuf - 1} steps (> the 129 MB L2)")
    cfg["launch"] = f"CUDA graphs of {args.nbuf} back-to-back steps (one per cache copy)"
    nb = args.nbuf

    # warm-up (also sets per-device kernel attributes before capture)
    for i in range(max(args.warmup, nb)):
        setup.step(i % nb)
    torch.cuda.synchronize()
    assert qs.device_error() == 0

    # one CUDA graph per cache copy
    s = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(s):
        for b in range(nb):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                setup.step(b)
            graphs.append(g)
    # the timed loop replays one graph of nb back-to-back steps (one per cache
    # copy, as a decode loop runs consecutive layers); a remainder of K % nb
    # steps uses the single-step graphs
    with torch.cuda.stream(s):
        g_run = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_run, stream=s):
            for b in range(nb):
                setup.step(b)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        graphs[i % nb].replay()
    g_run.replay()
    torch.cuda.synchronize()

    # timed region: exactly K steps
    K = args.steps
    reps, rem = divmod(K, nb)
    t_all = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_all[0].record()
        for i in range(reps):
            g_run.replay()
        for i in range(rem):
            graphs[i].replay()
        t_all[1].record()
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = t_all[0].elapsed_time(t_all[1])
    ms_per_step = total_ms / K
    ms_per_step = max_over_ranks(ms_per_step, dev)
    assert qs.device_error() == 0

    # the step-time distribution (after the timed region, not part of
    # `value`): the timed graph of nb back-to-back steps replayed between
    # two events, at least 200 times whatever --steps is; a sample is the
    # graph's time over nb (events between single steps would cut the
    # overlap of consecutive launches that the timed loop has)
    n_dist = max(200, min(reps, 2000))
    dist_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_dist)]
    torch.cuda.synchronize()
    for i in range(n_dist):
        dist_ev[i][0].record()
        g_run.replay()
        dist_ev[i][1].record()
    torch.cuda.synchronize()
    steps_us = sorted(a.elapsed_time(b) * 1e3 / nb for a, b in dist_ev)
    cfg["launch"] += f"; p50/p95 over {n_dist} replays of that graph (per step)"
    assert qs.device_error() == 0

    # per-stage device time of the unfused four-call path (each stage alone,
    # rotating copies, events); informational
    stage = {}
    for name, fn in (("append", setup.append), ("score", setup.score),
                     ("select", setup.select), ("attn", setup.attend),
                     ("unfused_step", setup.unfused), ("fused_step", setup.step)):
        stage[name] = time_stage(fn, nb, args.stage_reps) * 1e3
    by = setup.bytes()

    # e2e through the public API with host buffers
    e2e = run_e2e(setup, graphs, nb, args.e2e_steps)

    pk, pk_src = peaks()
    value = ms_per_step * 1e3
    path_gbs = by["total"] / (value * 1e-6) / 1e9
    # the timed region launches only the fused step kernel (the cluster
    # kernel or the grid-wide one, as the library plans this shape), back to
    # back on the replay stream: its average launch duration is the region's
    # time per step
    kname = qs.decode_step_kernel(len(setup.lens), w.h_kv, w.group, w.head_dim, w.page_size,
                                  w.dtype, setup.K, args.summary_fp8)
    dom_bytes = by["total"]
    dom_gbs = dom_bytes / (value * 1e-6) / 1e9
    traffic = ncu_traffic(kname, w.name + ("_e4m3" if args.summary_fp8 else ""))

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": data_desc(w),
        "config": cfg,
        "p50_us": round(steps_us[len(steps_us) // 2], 3),
        "p95_us": round(steps_us[int(len(steps_us) * 0.95)], 3),
        "stage_us": {k: round(v, 3) for k, v in stage.items()},
        "path": {"bytes": by["total"], "GBps": round(path_gbs, 1),
                 "frac": round(path_gbs / pk, 4), "frac_of_8TBps": round(path_gbs / 8000, 4)},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(dom_gbs, 1),
                     "peak": pk, "unit": "GB/s", "frac": round(dom_gbs / pk, 4),
                     "peak_source": pk_src, "bytes_per_launch": dom_bytes,
                     "traffic": traffic},
        "append_prefill": {**{k: round(v, 3) for k, v in setup.prefill.items()},
                           "frac": round(setup.prefill["GBps"] / pk, 4)},
        "e2e": e2e,
        "gpu_launches": K * LayerSetup.KERNELS_PER_STEP,
        "clocks": clk.summary(),
    }
    if args.gqa_union and w.group > 1:
        line["gqa_union"] = time_gqa_union(setup, args.stage_reps, pk, stage)
    if args.diagnostics > 0 and not args.summary_fp8:   # the diagnostics read kv-dtype summaries
        line["diagnostics"] = time_diagnostics(setup, args.diagnostics, args.stage_reps, pk)
    if rank == 0:
        if args.cpu_seconds > 0:
            line["cpu_baseline"] = cpu_baseline(setup, args.cpu_heads, args.cpu_seconds)
        print(json.dumps(line))


def run_model_step(args, w, cfg, dev, ws, rank, local):
    """A whole decode step of a multi-layer model: every layer has its own
    cache (prefilled through the library) and query; the first dense_layers
    layers attend over all pages (K = P), the others select with the budget.
    For each budget of the sweep, one CUDA graph holds the step's layers back
    to back; it is replayed and timed with events (each layer reads its own
    cold data: the layers together are far larger than L2). Per-layer times
    come from graphs of one dense and one sparse layer replayed alike."""
    import query_aware_sparse_gb300 as qs
    L = int(w.lengths()[0])
    S, h, d = w.page_size, w.h_kv, w.head_dim
    P = -(-L // S)
    t = wl.make_page_table([L], S, seed=w.seed)
    i32 = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32), device=dev)
    table = qs.PageTable(i32(t.page_indptr), i32(t.page_indices), i32([L]))
    pre = qs.PageTable(table.page_indptr, table.page_indices, i32([L - 1]))
    layers = []
    for layer in range(w.layers):
        k_tok, v_tok = wl.request_tokens(w, 0, L, layer=layer, device=dev)
        q = wl.queries(w, [L - 1], layer=layer, device=dev)
        kp, vp, sm = wl.empty_pool(t, h, d, w.dtype, device=dev, poison=False)
        cache = qs.PagedCache(kp, vp, sm)
        qs.append_kv(cache, pre, k_tok[:L - 1].contiguous(), v_tok[:L - 1].contiguous(),
                     i32([0, L - 1]), i32([0]))
        layers.append((cache, q, k_tok[L - 1:L].contiguous(), v_tok[L - 1:L].contiguous()))
        del k_tok, v_tok
    torch.cuda.synchronize()
    assert qs.device_error() == 0
    esz = torch.tensor([], dtype=w.dtype).element_size()
    pk, pk_src = peaks()

    def graph_of(calls):
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for c in calls:
                    c()
        return g, s

    def replay_us(g, s, reps):
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    sweep = {}
    whole_2048 = None
    for B in w.budgets:
        Ks = wl.selection_budget(B, S)
        steps = [qs.DecodeStep(c, table, w.group, P if i < w.dense_layers else Ks)
                 for i, (c, _, _, _) in enumerate(layers)]
        calls = [(lambda st=st, c=c, q=q, kn=kn, vn=vn: st(c, table, q, kn, vn))
                 for st, (c, q, kn, vn) in zip(steps, layers)]
        for c in calls:          # warm-up (kernel attributes before capture)
            c()
        torch.cuda.synchronize()
        assert qs.device_error() == 0
        g, s = graph_of(calls)
        reps = max(3, args.steps // w.layers)
        whole = replay_us(g, s, reps)
        nd = w.dense_layers
        gd, sd = graph_of(calls[:nd])                       # the dense layers
        dense_us = replay_us(gd, sd, max(3, args.stage_reps)) / max(nd, 1)
        ns = min(8, w.layers - nd)                          # distinct sparse layers
        gs_, ss = graph_of(calls[nd:nd + ns])
        sparse_us = replay_us(gs_, ss, max(3, args.stage_reps)) / ns
        summ = P * h * 2 * d * esz
        valid_sel = min(Ks, P) * S - (P * S - L if Ks >= P else 0)
        by_sparse = step_bytes(P, h, w.group, d, S, Ks, valid_sel, esz)["total"]
        by_dense = step_bytes(P, h, w.group, d, S, P, L, esz)["total"]
        by_whole = nd * by_dense + (w.layers - nd) * by_sparse
        sweep[str(B)] = {"k_pages": Ks, "whole_step_us": round(whole, 2),
                         "per_layer_us": round(whole / w.layers, 3),
                         "dense_layer_us": round(dense_us, 3),
                         "sparse_layer_us": round(sparse_us, 3),
                         "bytes_per_step": by_whole,
                         "GBps": round(by_whole / (whole * 1e-6) / 1e9, 1),
                         "frac": round(by_whole / (whole * 1e-6) / 1e9 / pk, 4),
                         "dense_summary_bytes_share": round(summ / by_dense, 4)}
        if B == 2048:
            whole_2048 = (whole, by_whole, reps)
        del g, gd, gs_, steps
    # the kernels the library plans for the sparse layers (the value's budget)
    # and for the dense ones (K = P)
    Kv = wl.selection_budget(2048 if whole_2048 else w.budgets[0], S)
    kname_sparse = qs.decode_step_kernel(1, h, w.group, d, S, w.dtype, Kv)
    kname_dense = qs.decode_step_kernel(1, h, w.group, d, S, w.dtype, P)
    whole, by_whole, reps = whole_2048 if whole_2048 else (
        sweep[str(w.budgets[0])]["whole_step_us"], sweep[str(w.budgets[0])]["bytes_per_step"], 1)
    per_layer = max_over_ranks(whole / w.layers, dev)
    cfg["budget_sweep_tokens"] = list(w.budgets)
    cfg["value_budget"] = 2048
    line = {"metric": METRIC, "value": round(per_layer, 3), "unit": UNIT, "n_gpus": ws,
            "steps": reps * w.layers, "warmup": args.warmup,
            "ms_per_step": round(per_layer / 1e3, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": data_desc(w),
            "config": cfg, "whole_step": sweep,
            "roofline": {"bound": "hbm", "kernel": kname_sparse, "dense_kernel": kname_dense,
                         "achieved": round(by_whole / (whole * 1e-6) / 1e9, 1), "peak": pk,
                         "unit": "GB/s", "frac": round(by_whole / (whole * 1e-6) / 1e9 / pk, 4),
                         "peak_source": pk_src, "bytes_per_launch": by_whole // w.layers,
                         "traffic": None},
            "gpu_launches": reps * w.layers}
    if rank == 0:
        if args.cpu_seconds > 0:
            v, v1, n, per = model_oracle(w, args.cpu_heads, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": round(v, 1), "unit": UNIT, "cores": n, "cores_1": round(v1, 1),
                "kind": "oracle", "layers_us": per,
                "sample": f"fp64 numpy oracle over layers {sorted(int(x) for x in per)} of the "
                          f"{w.layers} (dense: K = P; sparse: the 2048-token budget), every KV "
                          f"head on {n} single-threaded processes; the step is the dense layers' "
                          f"time plus the sparse layers' mean times {w.layers - w.dense_layers}, "
                          f"over {w.layers} layers; cores_1: {args.cpu_heads} heads on one core, "
                          f"scaled"}
        print(json.dumps(line))


def time_gqa_union(setup, reps, peak_gbs, stage):
    """GQA with a page set per query head (per-head scores, per-head Top-K,
    the per-KV-head union read once with head masks), as three calls, against
    the group-max path's separate calls on the same workload: device time per
    stage and the algorithmic bytes of each (summaries + K/V of the valid
    tokens of the pages read + q + o)."""
    qs, w = setup.qs, setup.w
    B, h, G, d, S, K = len(setup.lens), w.h_kv, w.group, w.head_dim, w.page_size, setup.K
    dev = setup.q.device
    h_q = h * G
    sc = torch.empty((h_q, setup.table_np.nnz), dtype=torch.float32, device=dev)
    sel = (torch.empty((B, h_q, K), dtype=torch.int32, device=dev),
           torch.empty((B, h_q, K), dtype=torch.int32, device=dev),
           torch.empty((B, h_q), dtype=torch.int32, device=dev))
    out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    un = (torch.empty((B, h, G * K), dtype=torch.int32, device=dev),
          torch.empty((B, h, G * K), dtype=torch.uint8, device=dev),
          torch.empty((B, h), dtype=torch.int32, device=dev))
    ws = torch.empty(max(qs.union_workspace_size(B, h, G, d, S, w.dtype, K), 16),
                     dtype=torch.uint8, device=dev)
    score = lambda b: qs.score_pages_per_head(setup.caches[b], setup.table, setup.q, G, sc)
    select = lambda b: qs.select_topk(setup.table, h_q, S, sc, K, out=sel)
    attend = lambda b: qs.union_decode_attn(setup.caches[b], setup.table, setup.q, G, sel[0], K,
                                            out, lse, union=un, workspace=ws)
    def whole(b):
        score(b)
        select(b)
        attend(b)
    t = {n: time_stage(f, len(setup.caches), reps) * 1e3
         for n, f in (("score", score), ("select", select), ("attn", attend), ("path", whole))}
    whole(0)
    assert qs.device_error() == 0
    ul = un[0].cpu().numpy()
    lens = setup.lens[:, None, None]
    valid = np.where(ul >= 0, np.clip(lens - ul.astype(np.int64) * S, 0, S), 0)
    esz = setup.k_dec.element_size()
    P = -(-setup.lens // S)
    summ = int(P.sum()) * h * 2 * d * setup.caches[0].summary.element_size()
    kv = int(valid.sum()) * 2 * d * esz
    qo_bytes = B * h_q * d * (esz + 4)
    gm = setup.bytes()
    total = summ + kv + qo_bytes
    return {"calls": "quest_score_pages_per_head + quest_select_topk (h_kv * group rows) + "
                     "quest_union_decode_attn",
            "us": {k: round(v, 3) for k, v in t.items()},
            "union_pages_per_unit": round(float(un[2].float().mean()), 1),
            "pages_per_unit_group_max": K,
            "bytes": total, "kv_bytes": kv, "GBps": round(total / (t["path"] * 1e-6) / 1e9, 1),
            "frac": round(total / (t["path"] * 1e-6) / 1e9 / peak_gbs, 4),
            "group_max_same_calls": {"us": round(stage["unfused_step"] - stage["append"], 3),
                                     "kv_bytes": gm["kv"]}}


def time_diagnostics(setup, R, reps, peak_gbs):
    """quest_recall_diagnostics (dense pass + reduction) on the workload with
    the fused step's latest selection: device time per call (one call per
    cache copy, so every call reads memory not touched by the previous one),
    its algorithmic bytes (every valid key and value, every page summary) and
    the diagnostics themselves, summarised over heads."""
    qs, w = setup.qs, setup.w
    sel = setup.fused.sel[0]
    nbuf = len(setup.caches)
    ws = torch.empty(max(qs.diag_workspace_size(w.h_kv, w.group, setup.table.nnz, w.page_size), 16),
                     dtype=torch.uint8, device=setup.q.device)
    fn = lambda b: qs.recall_diagnostics(setup.caches[b], setup.table, setup.q, w.group, sel,
                                         setup.K, R, workspace=ws)
    ms = time_stage(fn, nbuf, reps)
    d = fn(0)
    assert qs.device_error() == 0
    esz = setup.k_dec.element_size()
    P = -(-setup.lens // w.page_size)
    nbytes = int(2 * setup.lens.sum() * w.h_kv * w.head_dim * esz
                 + P.sum() * w.h_kv * 2 * w.head_dim * esz)
    slack = d["slack"].flatten()
    slack = slack[~torch.isnan(slack)]
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernels": "diag_pages_kernel + diag_reduce_kernel", "top_r": R,
            "us": round(ms * 1e3, 2), "bytes": nbytes, "GBps": round(gbs, 1),
            "frac": round(gbs / peak_gbs, 4),
            "eps_mean": float(d["eps"].mean()), "eps_max": float(d["eps"].max()),
            "topr_recall_mean": float(d["topr"].mean()), "topr_recall_min": float(d["topr"].min()),
            "slack_median": float(slack.median()), "vmax_max": float(d["vmax"].max())}


def run_e2e(setup, graphs, nb, n):
    """Same step through the public API with host buffers: each step copies
    q and the new token's k/v from pinned host memory, runs quest_decode_step
    and reads o and lse back into pinned host memory. q, k and v sit in one
    device buffer (and o and lse in another), so a step moves its inputs in
    one copy and its results in one; the upload, the step and the download are
    captured as one CUDA graph (one per cache copy), so a step is one graph
    launch and a synchronisation."""
    dev = setup.q.device

    def packed(ts):
        """One byte buffer holding the tensors back to back (16-B aligned
        parts) and views of it shaped like them."""
        sizes = [(t.nbytes + 15) // 16 * 16 for t in ts]
        buf = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
        views, off = [], 0
        for t, sz in zip(ts, sizes):
            views.append(buf[off:off + t.nbytes].view(t.dtype).view(t.shape))
            off += sz
        return buf, views

    d_in, (q, k1, v1) = packed([setup.q, setup.k_dec, setup.v_dec])
    q.copy_(setup.q)
    k1.copy_(setup.k_dec)
    v1.copy_(setup.v_dec)
    d_out, (o, lse) = packed([setup.fused.out, setup.fused.lse])
    h_in = d_in.cpu().pin_memory()
    h_out = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    fused = setup.fused
    saved = (fused.out, fused.lse)
    fused.out, fused.lse = o, lse            # the call writes its results into d_out
    s = torch.cuda.Stream()
    e2e = []
    try:
        with torch.cuda.stream(s):
            for b in range(nb):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    d_in.copy_(h_in, non_blocking=True)
                    fused(setup.caches[b], setup.table, q, k1, v1)
                    h_out.copy_(d_out, non_blocking=True)
                e2e.append(g)
        torch.cuda.synchronize()
        ts = []
        with torch.cuda.stream(s):               # replays go to s, the stream waited on
            for i in range(n + 10):
                t0 = time.perf_counter()
                e2e[i % nb].replay()
                s.synchronize()
                if i >= 10:
                    ts.append(time.perf_counter() - t0)
        ts.sort()
        assert torch.equal(h_out, d_out.cpu())
        hv = h_out[:o.nbytes].view(o.dtype).view(o.shape)
        setup.step(0)                            # the library's own buffers, same inputs
        torch.cuda.synchronize()
        assert torch.equal(hv, saved[0].cpu())
    finally:
        fused.out, fused.lse = saved
    bi = setup.q.nbytes + setup.k_dec.nbytes + setup.v_dec.nbytes
    bo = o.nbytes + lse.nbytes
    return {"value": round(statistics.median(ts) * 1e6, 3), "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "p95": round(ts[int(len(ts) * 0.95)] * 1e6, 3),
            "launch": "one CUDA graph per step: one upload of q, k and v from pinned memory, "
                      "the fused step, one download of o and lse to pinned memory; host waits "
                      "on each step"}


def oracle_timings(w, k_tok, v_tok, q, heads, seconds, n_sink=0, n_local=0, summary_fp8=False,
                   k=None, steps=None):
    """The oracle's decode step of one layer (request 0's inputs, every head),
    µs per layer (scaled to every request by pages): on one core over `heads`
    heads (scaled to all heads), and on every host core (one process per core,
    the KV heads split among them; at most one core per head). Each part takes
    about `seconds` (and at most `steps` samples, at least 3). Returns
    (one-core samples, all-core samples, cores used)."""
    def more(ts, t0):
        return len(ts) < 3 or (time.perf_counter() - t0 < seconds and
                               (steps is None or len(ts) < steps))

    h = min(heads, w.h_kv)
    one = OracleSample(w, k_tok[:, :h], v_tok[:, :h], q[:, :h * w.group], h, n_sink, n_local,
                       summary_fp8=summary_fp8, k=k)
    one.time_steps(1)
    t0 = time.perf_counter()
    ts1 = []
    while more(ts1, t0):
        ts1 += one.time_steps(1)
    del one
    n = min(host_cores(), w.h_kv)
    pool = OraclePool(n)
    try:
        pool.build(w, k_tok, v_tok, q, k=k, n_sink=n_sink, n_local=n_local,
                   summary_fp8=summary_fp8)
        # a round (every head once) on n cores, from the one-core figure
        est = statistics.median(ts1) * 1e-6 / pages_scale(w) / n
        per = max(1, int(0.1 / est)) if est > 0 else 1       # rounds per sample (~0.1 s)
        tsn, t0 = [], time.perf_counter()
        while more(tsn, t0):
            tsn.append(pool.time(per) * 1e6 * pages_scale(w))
    finally:
        pool.close()
    return ts1, tsn, n


def model_oracle(w, heads, seconds, layers=None):
    """The oracle's whole decode step of a multi-layer model, as µs per layer
    (the step over its layer count), from a stated subset of its layers:
    every dense layer of the subset (K = P) and its sparse layers (K of the
    2048-token budget) timed on every host core, each over all its KV heads
    and inputs regenerated from the layer's seed; the step is the dense
    layers' sum plus the sparse layers' mean times their count. On one core:
    `heads` heads of the first dense and first sparse layer, scaled."""
    L = int(w.lengths()[0])
    S = w.page_size
    P = -(-L // S)
    Ks = wl.selection_budget(2048, S)
    if layers is None:
        layers = sorted({0, w.dense_layers - 1, w.dense_layers, w.layers - 1} - {-1})
    n = min(host_cores(), w.h_kv)
    per, one = {}, {}
    pool = OraclePool(n)
    try:
        for layer in layers:
            k_tok, v_tok = wl.request_tokens(w, 0, L, layer=layer)
            q = wl.queries(w, [L - 1], layer=layer)[:1]
            dense = layer < w.dense_layers
            K = P if dense else Ks
            pool.build(w, k_tok, v_tok, q, k=K)
            ts, t0 = [], time.perf_counter()
            while len(ts) < 3 or time.perf_counter() - t0 < seconds / (2 * len(layers)):
                ts.append(pool.time(1) * 1e6)
            per[layer] = statistics.median(ts)
            if dense not in one:             # one core: a few heads of this kind of layer
                o = OracleSample(w, k_tok[:, :heads], v_tok[:, :heads], q[:, :heads * w.group],
                                 heads, k=K)
                o.time_steps(1)
                ts1, t0 = [], time.perf_counter()
                while len(ts1) < 3 or time.perf_counter() - t0 < seconds / 4:
                    ts1 += o.time_steps(1)
                one[dense] = statistics.median(ts1)
                del o
            del k_tok, v_tok
    finally:
        pool.close()
    dl = [per[x] for x in layers if x < w.dense_layers]
    sl = [per[x] for x in layers if x >= w.dense_layers]
    nd = w.dense_layers
    whole = (sum(dl) / max(len(dl), 1)) * nd + (sum(sl) / max(len(sl), 1)) * (w.layers - nd)
    whole1 = one.get(True, 0.0) * nd + one.get(False, 0.0) * (w.layers - nd)
    return whole / w.layers, whole1 / w.layers, n, {str(x): round(per[x], 1) for x in layers}


def cpu_baseline(setup, heads, seconds):
    ts1, tsn, n = oracle_timings(setup.w, *setup.sample, heads, seconds / 2, setup.n_sink,
                                 setup.n_local, summary_fp8=setup.summary_fp8)
    return {"value": round(statistics.median(tsn), 1), "unit": UNIT, "cores": n,
            "cores_1": round(statistics.median(ts1), 1), "kind": "oracle",
            "sample": f"fp64 numpy oracle decode step (append, score, select, attention) of "
                      f"request 0 of the same layer, scaled to every request by pages: on "
                      f"{n} cores ({n} single-threaded processes over the {setup.w.h_kv} KV "
                      f"heads, {len(tsn)} samples); cores_1: {min(heads, setup.w.h_kv)} of the heads "
                      f"on one core, scaled to all ({len(ts1)} steps)"}


def run_reference(args, w, cfg, dev, ws):
    """The oracle as the reference arm: same workload, metric and unit, on
    every host core (and on one, reported beside it)."""
    if w.layers > 1:
        v, v1, n, per = model_oracle(w, args.cpu_heads, 60.0)
        print(json.dumps({
            "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": ws, "steps": 1,
            "warmup": args.warmup, "ms_per_step": round(v * w.layers / 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg, "impl": "reference",
            "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": n,
                             "cores_1": round(v1, 1), "kind": "oracle", "layers_us": per,
                             "sample": f"layers {sorted(int(x) for x in per)}, every KV head, "
                                       f"on {n} single-threaded processes; per layer of the "
                                       f"{w.layers}-layer step"},
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return
    L = int(w.lengths()[0])
    k_tok, v_tok = wl.request_tokens(w, 0, L)
    q = wl.queries(w, [L - 1])[:1]
    # bounded: about a minute per part however many steps are asked
    ts1, tsn, n = oracle_timings(w, k_tok, v_tok, q, args.cpu_heads, 60.0, args.n_sink,
                                 args.n_local, summary_fp8=args.summary_fp8, steps=args.steps)
    v = statistics.median(tsn)
    line = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": ws,
            "steps": len(tsn), "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": cfg, "impl": "reference",
            "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": n,
                             "cores_1": round(statistics.median(ts1), 1), "kind": "oracle",
                             "sample": f"request 0 of the layer, every KV head, on {n} "
                                       f"single-threaded processes, scaled to every request by "
                                       f"pages; cores_1: {args.cpu_heads} heads on one core, "
                                       f"scaled"},
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
