"""The device entry points only enqueue work: no host synchronisation inside the library.

Right after pa_prefill_varlen (fused or not) / pa_decode return on the full-size Qwen2.5
workloads (hundreds of microseconds of GPU work), the stream must still have
work pending; a call that synchronised internally would return with the
stream idle.  (The packing and upload steps never read device memory either.)
"""
import time

import pytest
import torch

from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import dims_of

pytestmark = pytest.mark.gpu


def _pending_after(call):
    s = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    call()
    dt = time.perf_counter() - t0
    pending = not s.query()
    torch.cuda.synchronize()
    return pending, dt


def test_prefill_and_decode_calls_do_not_synchronise():
    wp = workloads.make("qwen25_prefill", device="cuda")
    bp = wp.batches[0]
    dims = dims_of(wp, bp)
    plan = pa.pa_pack_prefill(dims, bp.seq_lens, bp.query_lens, bp.block_lists).upload()
    pa.pa_store_kvcache(dims, bp.k, bp.v, wp.pool.k_cache, wp.pool.v_cache, plan.slot_mapping, bp.num_tokens)
    out = torch.empty_like(bp.q)
    call = lambda: [pa.pa_prefill_varlen(dims, bp.q, wp.pool.k_cache, wp.pool.v_cache, plan, bp.scale, out)
                    for _ in range(3)]
    call()
    pending, dt = _pending_after(call)
    assert pending, f"prefill calls returned with the stream idle ({dt * 1e3:.2f} ms)"

    kc, vc = wp.pool.k_cache.clone(), wp.pool.v_cache.clone()
    call = lambda: [pa.pa_prefill_varlen_fused(dims, bp.q, bp.k, bp.v, kc, vc, plan, bp.scale, out)
                    for _ in range(3)]
    call()
    pending, dt = _pending_after(call)
    assert pending, f"fused store + prefill calls returned with the stream idle ({dt * 1e3:.2f} ms)"

    wd = workloads.make("qwen25_decode", device="cuda")
    bd = wd.batches[0]
    dims = dims_of(wd, bd)
    dplan = pa.pa_pack_decode(dims, bd.seq_lens, bd.block_lists).upload()
    ws = pa.decode_workspace(dplan)
    out = torch.empty_like(bd.q)
    call = lambda: [pa.pa_decode(dims, bd.q, wd.pool.k_cache, wd.pool.v_cache, dplan, bd.scale, out, ws)
                    for _ in range(3)]
    call()
    pending, dt = _pending_after(call)
    assert pending, f"decode calls returned with the stream idle ({dt * 1e3:.2f} ms)"
