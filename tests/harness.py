"""Run a workload through libpagedattn (GPU) and through the CPU oracle.

Both sides receive the same seeded inputs from ``workloads``; each computes
its own metadata (the library through pa_pack_*, the oracle through its own
slot mapping) and its own result.  Nothing the GPU produces feeds the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa

MAX_ABS = 2e-2   # |o_gpu - o_ref| bound (bf16 inputs, fp32 accumulation)
MAX_RRMS = 1e-2  # ||o_gpu - o_ref||_2 / ||o_ref||_2


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def dims_of(w, batch) -> pa.pa_dims:
    p = w.pool
    return pa.make_dims(p.num_blocks, p.block_size, batch.num_heads, p.num_kv_heads, p.head_dim)


def run_gpu_batch(w, batch, k_cache, v_cache, split_tokens: int = 0, stream=None):
    """Store the batch's new K/V, then prefill or decode. Returns out (bf16, device)."""
    dims = dims_of(w, batch)
    dev = k_cache.device
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    out = torch.empty_like(q)
    if batch.kind == "prefill":
        plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload(dev, stream)
        pa.pa_store_kvcache(dims, k, v, k_cache, v_cache, plan.slot_mapping, batch.num_tokens, stream=stream)
        pa.pa_prefill_varlen(dims, q, k_cache, v_cache, plan, batch.scale, out, stream=stream)
    else:
        plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split_tokens).upload(dev, stream)
        pa.pa_store_kvcache(dims, k, v, k_cache, v_cache, plan.slot_mapping, batch.num_tokens, stream=stream)
        ws = pa.decode_workspace(plan, dev)
        pa.pa_decode(dims, q, k_cache, v_cache, plan, batch.scale, out, ws, stream=stream)
    return out, plan


def compare(out_gpu: torch.Tensor, ref: np.ndarray, rows=None):
    """Max-abs and relative-RMS errors of the GPU output (bf16) against the fp64 oracle."""
    got = out_gpu.detach().to(torch.float64).cpu().numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.sqrt((ref ** 2).sum()))
    rrms = float(np.sqrt((diff ** 2).sum()) / denom) if denom > 0 else float(np.sqrt((diff ** 2).sum()))
    return max_abs, rrms


def assert_close(out_gpu, ref, rows=None, what=""):
    assert np.isfinite(out_gpu.detach().float().cpu().numpy()).all(), f"{what}: non-finite output"
    max_abs, rrms = compare(out_gpu, ref, rows)
    print(f"[parity] {what}: max|err|={max_abs:.3e} (bound {MAX_ABS}) rel-rms={rrms:.3e} (bound {MAX_RRMS})")
    assert max_abs <= MAX_ABS and rrms <= MAX_RRMS, f"{what}: max|err|={max_abs:.3e} rel-rms={rrms:.3e}"
    return max_abs, rrms


def sample_rows(batch, per_seq: int, seed: int = 0) -> np.ndarray:
    """Query rows to check at full size: first, last and random rows of each sequence."""
    rng = np.random.default_rng(seed)
    sel = np.zeros(batch.num_tokens, dtype=bool)
    t0 = 0
    for lq in batch.query_lens:
        lq = int(lq)
        if lq:
            idx = {0, lq - 1} | set(rng.integers(0, lq, size=min(per_seq, lq)).tolist())
            sel[[t0 + i for i in idx]] = True
        t0 += lq
    return sel


def oracle_subset_pool(pool_k: torch.Tensor, pool_v: torch.Tensor, batch, seqs):
    """Host copies of only the blocks the selected sequences use, block ids relabelled.

    Input preparation for the oracle on pools too large to copy whole; the
    oracle's output is invariant under block relabelling (pinned on the CPU).
    """
    used = np.unique(np.concatenate([batch.block_lists[b] for b in seqs]))
    remap = {int(p): i for i, p in enumerate(used)}
    idx = torch.from_numpy(used.astype(np.int64)).to(pool_k.device)
    sub_k = bits(pool_k.index_select(0, idx))
    sub_v = bits(pool_v.index_select(0, idx))
    lists = [np.array([remap[int(p)] for p in batch.block_lists[b]], np.int32) for b in seqs]
    return sub_k, sub_v, lists


def int8_pools(w, num_heads: int):
    """Quantise the workload's bf16 pool on both sides, independently.

    GPU: pa_store_kvcache_int8 over every slot of the pool.  Oracle:
    oracle.quantize_rows on a host copy, scales moved to the cache's
    head-major [blocks][kv heads][block] layout.  Returns (gpu, host) tuples
    of (k_codes, v_codes, k_scale, v_scale); host scales are fp16 bits.
    """
    p = w.pool
    dev = p.k_cache.device
    dims = pa.make_dims(p.num_blocks, p.block_size, num_heads, p.num_kv_heads, p.head_dim)
    n = p.num_blocks * p.block_size
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    gpu = pa.int8_cache(dims, dev)
    pa.pa_store_kvcache_int8(dims, p.k_cache.view(n, p.num_kv_heads, p.head_dim),
                             p.v_cache.view(n, p.num_kv_heads, p.head_dim), *gpu, slots, n)
    kc, ks = oracle.quantize_rows(p.k_cache.cpu())
    vc, vs = oracle.quantize_rows(p.v_cache.cpu())
    host = (kc, vc, np.ascontiguousarray(ks.transpose(0, 2, 1)), np.ascontiguousarray(vs.transpose(0, 2, 1)))
    return gpu, host


def int8_equal(gpu, host, what=""):
    """Bit-exact comparison of a GPU INT8 cache with the oracle's."""
    names = ("k codes", "v codes", "k scales", "v scales")
    for name, g, h in zip(names, gpu, host):
        got = g.cpu().numpy()
        if got.dtype == np.float16:
            got = got.view(np.uint16)
        bad = np.count_nonzero(got != h)
        assert bad == 0, f"{what}: {bad} of {h.size} {name} differ"


def run_gpu_batch_int8(w, batch, cache, split_tokens: int = 0, stream=None):
    """Quantising store of the batch's new K/V, then INT8 prefill or decode. Returns (out, plan)."""
    if batch.kind == "decode":
        return run_gpu_decode_int8(w, batch, cache, split_tokens, stream)
    dims = dims_of(w, batch)
    dev = cache[0].device
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    out = torch.empty_like(q)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload(dev, stream)
    pa.pa_store_kvcache_int8(dims, k, v, *cache, plan.slot_mapping, batch.num_tokens, stream=stream)
    pa.pa_prefill_varlen_int8(dims, q, *cache, plan, batch.scale, out, stream=stream)
    return out, plan


def run_gpu_decode_int8(w, batch, cache, split_tokens: int = 0, stream=None):
    """Quantising store of the batch's new K/V, then INT8 decode. Returns out (bf16, device)."""
    dims = dims_of(w, batch)
    dev = cache[0].device
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    out = torch.empty_like(q)
    plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split_tokens).upload(dev, stream)
    pa.pa_store_kvcache_int8(dims, k, v, *cache, plan.slot_mapping, batch.num_tokens, stream=stream)
    ws = pa.decode_workspace(plan, dev)
    pa.pa_decode_int8(dims, q, *cache, plan, batch.scale, out, ws, stream=stream)
    return out, plan
