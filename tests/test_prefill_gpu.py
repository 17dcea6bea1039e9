"""Prefill parity against the fp64 oracle: max |err| <= 2e-2, relative RMS <= 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, bits, dims_of, run_gpu_batch, sample_rows

pytestmark = pytest.mark.gpu


def _run_both(w, batch_idx=None, row_select=None):
    """Run every batch in order on both sides; return the outputs of the chosen batch."""
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    res = []
    for i, batch in enumerate(w.batches):
        out, _ = run_gpu_batch(w, batch, kc, vc)
        ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size, row_select=row_select)
        res.append((batch, out, ref))
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    return res if batch_idx is None else res[batch_idx]


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefill_32", "qwen3_prefill_128", "qwen3_prefill_256",
                                  "qwen3_prefix", "qwen3_chunked"])
def test_prefill_configs(name):
    w = workloads.make(name, device="cuda")
    for batch, out, ref in _run_both(w):
        if batch.kind == "prefill":
            assert_close(out, ref, what=name)


# random ragged cases: several tiles and a ragged tail, every supported shape class
CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (101, 3, 2, 1, 64, 16, 300, None),
    (102, 4, 4, 2, 64, 256, 700, "random"),
    (103, 5, 7, 1, 128, 16, 400, "random"),
    (104, 3, 14, 2, 128, 256, 520, None),
    (105, 6, 8, 8, 128, 16, 260, "random"),
    (106, 2, 16, 1, 64, 32, 390, "random"),
    (107, 4, 28, 4, 128, 16, 333, "random"),
    (108, 3, 16, 8, 128, 1024, 1100, "random"),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_prefill_random(case):
    seed, B, hq, hkv, d, bs, max_len, cached = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, device="cuda",
                              cached=cached)
    batch, out, ref = _run_both(w, 0)
    assert_close(out, ref, what=f"case {seed}")


# Many more work items than SMs: every CTA of the persistent kernel runs several
# items back to back (rings, barrier phases, tail zeroing and query refills
# carried across items; empty second query tiles; prefix and no-prefix items).
MULTI = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (121, 160, 4, 4, 128, 16, 512, "random"),
    (122, 96, 16, 4, 64, 32, 300, "random"),
    (123, 48, 28, 4, 128, 16, 200, None),
    (124, 200, 16, 8, 128, 256, 300, "random"),
]


@pytest.mark.parametrize("case", MULTI, ids=[str(c[0]) for c in MULTI])
def test_prefill_many_items_per_cta(case):
    seed, B, hq, hkv, d, bs, max_len, cached = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, device="cuda",
                              cached=cached)
    b = w.batches[0]
    items = pa.pa_pack_prefill(dims_of(w, b), b.seq_lens, b.query_lens, b.block_lists, pin=False).meta.num_tiles
    assert items > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    batch, out, ref = _run_both(w, 0)
    assert_close(out, ref, what=f"case {seed}, {items} items")


def test_prefill_output_alignment_16_and_32_bytes():
    """An output 16 but not 32 bytes aligned (allowed) gives the same bits as an aligned one."""
    w = workloads.random_case(131, num_seqs=40, hq=8, hkv=2, d=128, bs=16, max_len=400, device="cuda")
    b = w.batches[0]
    dims = dims_of(w, b)
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    plan = pa.pa_pack_prefill(dims, b.seq_lens, b.query_lens, b.block_lists).upload("cuda")
    q, k, v = b.q.cuda(), b.k.cuda(), b.v.cuda()
    pa.pa_store_kvcache(dims, k, v, kc, vc, plan.slot_mapping, b.num_tokens)
    out32 = torch.empty_like(q)
    assert out32.data_ptr() % 32 == 0
    buf = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
    out16 = buf[8:].view(q.shape)  # 16 bytes past a 32-byte boundary
    assert out16.data_ptr() % 32 == 16
    pa.pa_prefill_varlen(dims, q, kc, vc, plan, b.scale, out32)
    pa.pa_prefill_varlen(dims, q, kc, vc, plan, b.scale, out16)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert np.array_equal(bits(out32), bits(out16))


def test_prefill_edge_lengths():
    """Sequences with no new tokens, single-token sequences and a 1-of-N suffix in one batch."""
    hq, hkv, d, bs = 4, 2, 64, 16
    lens = np.array([1, 17, 40, 129, 5, 64], np.int32)
    qlens = np.array([1, 0, 1, 129, 0, 64], np.int32)
    nb = int(sum(-(-l // bs) for l in lens)) + 2
    perm = np.random.default_rng(7).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(8)
    mk = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = int(qlens.sum())
    batch = workloads.Batch("prefill", lens, qlens, blocks, mk(t, hq, d), mk(t, hkv, d), mk(t, hkv, d), hq, d ** -0.5)
    w = workloads.Workload("edges", pool, [batch])
    batch, out, ref = _run_both(w, 0)
    assert_close(out, ref, what="edges")


def test_prefill_empty_batch_is_a_no_op():
    dims = pa.make_dims(4, 16, 2, 1, 64)
    plan = pa.pa_pack_prefill(dims, [5, 3], [0, 0], [[0], [1]]).upload()
    assert plan.meta.num_tiles == 0
    q = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_prefill_varlen(dims, q, kc, kc, plan, 0.125, q)
    torch.cuda.synchronize()


def test_prefill_permutation_invariance_bitwise():
    """Relabelling physical blocks (pool contents moved with them) changes nothing, bit for bit."""
    w = workloads.random_case(111, num_seqs=3, hq=4, hkv=2, d=128, bs=16, max_len=300, device="cuda")
    batch = w.batches[0]
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    out_a, _ = run_gpu_batch(w, batch, kc, vc)
    nb = w.pool.num_blocks
    sigma = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(sigma)
    inv[sigma] = torch.arange(nb)
    w2 = workloads.Workload("perm", workloads.Pool(nb, w.pool.block_size, w.pool.num_kv_heads, w.pool.head_dim,
                                                   w.pool.k_cache[inv.cuda()].clone(),
                                                   w.pool.v_cache[inv.cuda()].clone()), [])
    b2 = workloads.Batch(batch.kind, batch.seq_lens, batch.query_lens,
                         [sigma.numpy()[b].astype(np.int32) for b in batch.block_lists],
                         batch.q, batch.k, batch.v, batch.num_heads, batch.scale)
    out_b, _ = run_gpu_batch(w2, b2, w2.pool.k_cache, w2.pool.v_cache)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)


def test_prefix_suffix_equals_full_prefill_rows_on_gpu():
    """Prefix-cache hit (44 new of 300) reproduces rows 256..299 of the full prefill."""
    g = torch.Generator(device="cuda").manual_seed(9)
    mk = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(4, 256, 8, 128, mk(4, 256, 8, 128), mk(4, 256, 8, 128))
    q, k, v = mk(300, 16, 128), mk(300, 8, 128), mk(300, 8, 128)
    full = workloads.Batch("prefill", np.array([300], np.int32), np.array([300], np.int32),
                           [np.array([2, 0], np.int32)], q, k, v, 16, 128 ** -0.5)
    wf = workloads.Workload("full", pool, [full])
    kc, vc = pool.k_cache.clone(), pool.v_cache.clone()
    out_full, _ = run_gpu_batch(wf, full, kc, vc)
    sfx = workloads.Batch("prefill", np.array([300], np.int32), np.array([44], np.int32),
                          [np.array([2, 0], np.int32)], q[256:].contiguous(), k[256:].contiguous(),
                          v[256:].contiguous(), 16, 128 ** -0.5)
    out_sfx, _ = run_gpu_batch(wf, sfx, kc, vc)
    torch.cuda.synchronize()
    ref = out_full[256:].double().cpu().numpy()
    assert_close(out_sfx, ref, what="suffix vs full")


def test_prefill_qwen25_full_size_every_row():
    """4 x 4096, Hq 28 / Hkv 4, block 16 (the benched prompt batch): the full launch against
    the oracle on every query row and head."""
    w = workloads.make("qwen25_prefill", device="cuda")
    batch = w.batches[0]
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    out, _ = run_gpu_batch(w, batch, kc, vc)
    ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert_close(out, ref, what="qwen25 prefill (every row)")


def test_prefill_single_32k_sequence_sampled_rows():
    """One 32768-token causal prompt (Qwen2.5 heads): items of up to 256 key tiles, so every
    ring and the release-event ring wrap many times within an item; oracle on sampled rows."""
    w = workloads.random_case(161, num_seqs=1, hq=28, hkv=4, d=128, bs=16, min_len=32768, max_len=32768,
                              cached=None, device="cuda")
    batch = w.batches[0]
    sel = sample_rows(batch, per_seq=24, seed=7)
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    out, _ = run_gpu_batch(w, batch, kc, vc)
    ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size, row_select=sel)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert_close(out, ref, rows=sel, what="single 32k prefill")
    assert torch.isfinite(out.float()).all()


def test_mixed_prefill_and_decode_rows_in_one_launch():
    """Decode rows are prefill rows with one query token: one varlen launch serves a mixed batch
    (long-context single-token rows next to full prompts and cached-prefix suffixes)."""
    hq, hkv, d, bs = 28, 4, 128, 16
    lens = np.array([3000, 1, 700, 2048, 129, 999, 4096], np.int32)
    qlens = np.array([1, 1, 700, 1, 60, 1, 300], np.int32)
    nb = int(sum(-(-l // bs) for l in lens)) + 5
    perm = np.random.default_rng(17).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(18)
    mk = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = int(qlens.sum())
    batch = workloads.Batch("prefill", lens, qlens, blocks, mk(t, hq, d), mk(t, hkv, d), mk(t, hkv, d), hq, d ** -0.5)
    w = workloads.Workload("mixed", pool, [batch])
    batch, out, ref = _run_both(w, 0)
    assert_close(out, ref, what="mixed prefill+decode")
