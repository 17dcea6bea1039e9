"""pa_decode_static: decode for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace (for example code
running while a stream is captured into a CUDA graph, where cudaMalloc is not
allowed, or runtimes that only own fixed pre-planned buffers).  For them
pa_decode_static uses the library's own fixed scratch array instead.  These
tests call it through the C ABI and check it against pa_decode (which gets a
caller workspace) and against the CPU oracle, on two calls in a row because the
array is shared and keeps the previous call's contents.  The file is named so
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import MAX_ABS, MAX_RRMS, assert_close, bits, compare, dims_of

pytestmark = pytest.mark.gpu


def _setup(seed, split):
    w = workloads.random_case(seed, num_seqs=6, hq=14, hkv=2, d=128, bs=16, max_len=3000, min_len=1000,
                              kind="decode", device="cuda")
    batch = w.batches[0]
    dims = dims_of(w, batch)
    plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split_tokens=split).upload()
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    pa.pa_store_kvcache(dims, batch.k, batch.v, kc, vc, plan.slot_mapping, batch.num_tokens)
    return w, batch, dims, plan, kc, vc


def test_static_scratch_matches_workspace_decode_twice():
    w, batch, dims, plan, kc, vc = _setup(301, 256)
    assert plan.meta.num_partials > 0  # the scratch really is used
    assert 0 < plan.meta.workspace_bytes <= pa.PA_DECODE_STATIC_SCRATCH_BYTES
    ref = torch.empty_like(batch.q)
    pa.pa_decode(dims, batch.q, kc, vc, plan, batch.scale, ref, pa.decode_workspace(plan))
    torch.cuda.synchronize()
    ref64 = ref.double().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(batch.q, float("nan"))
        pa.pa_decode_static(dims, batch.q, kc, vc, plan, batch.scale, out)
        torch.cuda.synchronize()
        max_abs, rrms = compare(out, ref64)
        assert max_abs <= MAX_ABS and rrms <= MAX_RRMS, (max_abs, rrms)


def test_static_scratch_matches_the_oracle_twice():
    """Against the fp64 CPU oracle (its own store of the batch, then attention), two calls in a row."""
    w, batch, dims, plan, kc, vc = _setup(305, 256)
    assert plan.meta.num_partials > 0
    ref, _ = oracle.run_batch(bits(w.pool.k_cache), bits(w.pool.v_cache), batch, w.pool.block_size)
    for i in range(2):
        out = torch.full_like(batch.q, float("nan"))
        pa.pa_decode_static(dims, batch.q, kc, vc, plan, batch.scale, out)
        torch.cuda.synchronize()
        assert_close(out, ref, what=f"pa_decode_static call {i + 1}")


def test_static_scratch_second_plan_after_first():
    """A different plan after another one: leftover scratch contents must not leak into the result."""
    for seed, split in ((302, 512), (303, 128)):
        w, batch, dims, plan, kc, vc = _setup(seed, split)
        ref = torch.empty_like(batch.q)
        pa.pa_decode(dims, batch.q, kc, vc, plan, batch.scale, ref, pa.decode_workspace(plan))
        out = torch.empty_like(batch.q)
        pa.pa_decode_static(dims, batch.q, kc, vc, plan, batch.scale, out)
        torch.cuda.synchronize()
        max_abs, rrms = compare(out, ref.double().cpu().numpy())
        assert max_abs <= MAX_ABS and rrms <= MAX_RRMS, (seed, max_abs, rrms)


def test_static_scratch_rejects_plans_beyond_its_size():
    w, batch, dims, plan, kc, vc = _setup(304, 256)
    big = pa.pa_decode_meta.from_buffer_copy(plan.meta)
    big.workspace_bytes = pa.PA_DECODE_STATIC_SCRATCH_BYTES + 256
    out = torch.empty_like(batch.q)
    rc = pa.lib().pa_decode_static(ctypes.byref(dims), batch.q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                   plan.dptr(plan.meta.off_context_lens), plan.dptr(plan.meta.off_block_tables),
                                   ctypes.c_float(batch.scale), out.data_ptr(), ctypes.byref(big),
                                   plan.dptr(plan.meta.off_items), plan.dptr(plan.meta.off_seq_items),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_WORKSPACE
    assert "scratch" in pa.pa_last_error_string()
