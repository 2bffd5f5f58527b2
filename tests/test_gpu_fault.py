"""Failure handling of the kernels' bounded waits, made to run out on purpose
through the library's test hook (quest_test_step_fault): a wait on a barrier
that nothing arrives on (the fused step on clusters) and a copy slot that
expects more bytes than its copies bring (the split-K attention). The call
must come back with QUEST_DEVERR_WAIT_TIMEOUT in the device error word and
leave the device usable: the next normal call passes parity against the
oracle. No fault, trap or endless loop is involved: every wait gives up after
a few thousand tries."""

import numpy as np
import pytest
import torch

from oracle import quest_oracle as qo
from tests._cases import F16, attn_close, dev_i32, gpu_cache, gpu_table, np_of, random_case
from tests.test_gpu_step import _run, _w

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 0x8
LIMIT = 2000                  # tries per wait (each up to about 1 us)


@pytest.mark.parametrize("batch,h_kv,group,lens_fn", [
    (1, 4, 1, lambda: [5000]),                                # one unit per cluster
    (24, 8, 1, lambda: list(range(40, 40 + 24 * 37, 37))),    # several units per cluster
    (3, 2, 4, lambda: [900, 17, 3000]),                       # GQA on the warp MMA
])
def test_step_wait_runs_out_then_next_call_passes(batch, h_kv, group, lens_fn):
    import query_aware_sparse_gb300 as qs
    lens = lens_fn()
    k = 16
    assert qs.decode_step_kernel(batch, h_kv, group, 64, 16, F16, k) == "cstep_kernel"
    case = random_case(90 + batch, lens, h_kv=h_kv, group=group, d=64, S=16, dtype=F16)
    t = case["table"]
    sm = qo.build_summary(np_of(case["k_pool"]), t.page_indptr, t.page_indices, t.seq_lens,
                          summary=np_of(case["summary"]))
    cache = gpu_cache(case["k_pool"], case["v_pool"], torch.from_numpy(sm))
    table = gpu_table(t)
    step = qs.DecodeStep(cache, table, group, k)
    qs.device_error()                       # start from a clear error word
    qs.test_step_fault(1, LIMIT)
    try:
        step(cache, table, case["q"].cuda())
        err = qs.device_error()
    finally:
        qs.test_step_fault(0, 0)
    assert err & WAIT_TIMEOUT, err
    # the same process and context: a normal multi-step run matches the oracle
    _run(_w("after_fault", batch=batch, h_kv=h_kv, group=group, head_dim=64, k=k),
         lens, steps=2, seed=95 + batch)


def _sets(case, k):
    t = case["table"]
    sl = np.full((t.batch, case["h_kv"], k), -1, np.int32)
    for r in range(t.batch):
        P = -(-int(t.seq_lens[r]) // t.page_size)
        n = min(P, k)
        sl[r, :, :n] = np.arange(n)
    sp = np.where(sl >= 0, t.page_indices[np.maximum(sl, 0) + t.page_indptr[:-1, None, None]], -1)
    return sl, sp.astype(np.int32)


@pytest.mark.parametrize("entry", ["workspace", "noalloc"])
def test_attention_wait_runs_out_then_next_call_passes(entry):
    import ctypes
    import query_aware_sparse_gb300 as qs
    group, k = 2, 48
    case = random_case(97, [2000, 300, 40], h_kv=2, group=group, d=128, S=16, dtype=F16)
    t = case["table"]
    cache = gpu_cache(case["k_pool"], case["v_pool"], case["summary"])
    table = gpu_table(t)
    sl, sp = _sets(case, k)
    q = case["q"].cuda()

    def call():
        if entry == "workspace":
            return qs.sparse_decode_attn(cache, table, q, group, dev_i32(sl), dev_i32(sp), k)
        B, h_q, d = q.shape
        out = torch.empty((B, h_q, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, h_q), dtype=torch.float32, device="cuda")
        sld, spd = dev_i32(sl), dev_i32(sp)
        st = qs.lib().quest_sparse_decode_attn_noalloc(
            ctypes.byref(cache.c), ctypes.byref(table.c), q.data_ptr(), group, sld.data_ptr(),
            spd.data_ptr(), k, out.data_ptr(), lse.data_ptr(), ctypes.c_float(0.0),
            torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        return out, lse

    qs.device_error()
    qs.test_step_fault(2, LIMIT)
    try:
        call()
        err = qs.device_error()
    finally:
        qs.test_step_fault(0, 0)
    assert err & WAIT_TIMEOUT, err
    o, lse = call()
    assert qs.device_error() == 0
    ro, rl = qo.sparse_attention(np_of(case["q"]), np_of(case["k_pool"]), np_of(case["v_pool"]),
                                 t.page_indptr, t.page_indices, t.seq_lens, sl, group)
    ok, rel = attn_close(np_of(o), ro)
    assert ok.all(), rel.max()
    assert np.all(np.abs(np_of(lse) - rl) <= 1e-3 * np.maximum(1, np.abs(rl)))


def test_fault_hook_rejects_unknown_modes():
    import query_aware_sparse_gb300 as qs
    assert qs.lib().quest_test_step_fault(3, 0) != 0
    assert qs.lib().quest_test_step_fault(1, -1) != 0
    assert qs.lib().quest_test_step_fault(0, 0) == 0
