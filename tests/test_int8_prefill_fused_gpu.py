"""pa_prefill_varlen_int8_fused (quantising store of the new tokens + INT8 prefill in one call).

Checked three ways: the whole INT8 cache (codes and fp16 scales) after every
call equals the oracle's store bit for bit; the output is within the oracle
tolerance (max |err| <= 2e-2, relative RMS <= 1e-2) of the oracle's attention
over its own dequantised cache; and it is bitwise the output of
pa_store_kvcache_int8 + pa_prefill_varlen_int8 run on a second copy of the
cache (the gather launch quantises the new rows with the store's arithmetic
and dequantises those codes with the stored fp16 scale, which is what the
unfused gather reads back from the cache).

Method: "面试问答准备: nano-vLLM 推理引擎优化", Q3 (INT8 cache: codes + fp16
scale per token and head; the prefill's extra cost sits outside the attention
kernel) and "手搓 vLLM 推理引擎", Step 4 (store the new K/V, then attend over
the cache).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, dims_of, int8_equal, int8_pools, run_gpu_batch_int8

pytestmark = pytest.mark.gpu


def _fused(w, batch, cache, plan=None):
    dims = dims_of(w, batch)
    dev = cache[0].device
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    if plan is None:
        plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload(dev)
    out = torch.full_like(q, float("nan"))
    pa.pa_prefill_varlen_int8_fused(dims, q, k, v, *cache, plan, batch.scale, out)
    return out, plan


def _run(w, row_select=None):
    """Every batch in order: prefill batches through the fused call (decode batches through the
    store + INT8 decode), the separate two-launch path on a second cache, the oracle alongside."""
    gpu, host = int8_pools(w, w.batches[0].num_heads)
    gpu2 = tuple(t.clone() for t in gpu)
    res = []
    for batch in w.batches:
        if batch.kind == "prefill":
            out, plan = _fused(w, batch, gpu)
        else:
            out, plan = run_gpu_batch_int8(w, batch, gpu)
        sep, _ = run_gpu_batch_int8(w, batch, gpu2)
        sel = row_select(batch) if callable(row_select) else row_select
        ref, _ = oracle.run_batch_int8(*host, batch, w.pool.block_size, row_select=sel)
        res.append((batch, out, sep, ref, plan))
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(gpu, host, what=f"{w.name} (fused)")
    for a, b in zip(gpu, gpu2):
        assert torch.equal(a, b), f"{w.name}: fused cache differs from store_int8's"
    return res


def _check(res, what):
    for batch, out, sep, ref, _ in res:
        assert_close(out, ref, what=f"{what} {batch.kind}")
        assert torch.equal(out, sep), f"{what} {batch.kind}: fused output differs from store_int8 + prefill_int8"


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefill_32", "qwen3_prefill_128", "qwen3_prefill_256",
                                  "qwen3_prefix", "qwen3_chunked"])
def test_int8_fused_prefill_configs(name):
    _check(_run(workloads.make(name, device="cuda")), f"int8 fused {name}")


CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (801, 3, 2, 1, 64, 16, 300, None),
    (802, 4, 4, 2, 64, 256, 700, "random"),
    (803, 5, 7, 1, 128, 16, 400, "random"),
    (804, 3, 14, 2, 128, 256, 520, None),
    (805, 6, 8, 8, 128, 16, 260, "random"),       # 8 KV heads
    (806, 2, 16, 1, 64, 32, 390, "random"),
    (807, 4, 28, 4, 128, 16, 333, "random"),
    (808, 3, 16, 8, 128, 1024, 1100, "random"),
    (809, 160, 4, 4, 128, 16, 512, "random"),     # many items per CTA
    (810, 96, 16, 4, 64, 32, 300, "random"),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_int8_fused_prefill_random(case):
    seed, ns, hq, hkv, d, bs, ml, cached = case
    w = workloads.random_case(seed, num_seqs=ns, hq=hq, hkv=hkv, d=d, bs=bs, max_len=ml, cached=cached,
                              device="cuda")
    _check(_run(w), f"int8 fused case {seed}")


def test_int8_fused_prefill_qwen25_every_row():
    """The benched 4 x 4096 prompt batch, every output row against the oracle."""
    _check(_run(workloads.make("qwen25_prefill", device="cuda")), "int8 fused qwen25 prefill")


def test_int8_fused_prefill_edge_lengths():
    """Sequences without new tokens, single tokens, exact tiles and unaligned prefixes in one batch."""
    hq, hkv, d, bs = 4, 2, 128, 16
    lens = np.array([16, 17, 48, 129, 5, 128, 256, 77], np.int32)
    qlens = np.array([0, 1, 16, 129, 0, 128, 96, 30], np.int32)  # prefixes 16, 16, 32, 0, -, 0, 160, 47
    nb = int(sum(-(-int(l) // bs) for l in lens)) + 2
    perm = np.random.default_rng(29).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(30)
    mk = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = int(qlens.sum())
    batch = workloads.Batch("prefill", lens, qlens, blocks, mk(t, hq, d), mk(t, hkv, d), mk(t, hkv, d), hq, d ** -0.5)
    _check(_run(workloads.Workload("int8_fused_edges", pool, [batch])), "int8 fused edges")


def test_int8_fused_prefill_plan_launched_again():
    """One uploaded plan and one workspace used three times: every call gives the same output and
    leaves the same cache (the new rows are stored again with the same codes and scales)."""
    w = workloads.random_case(821, num_seqs=40, hq=8, hkv=2, d=128, bs=16, max_len=700, cached="random",
                              device="cuda")
    batch = w.batches[0]
    gpu, _ = int8_pools(w, batch.num_heads)
    dims = dims_of(w, batch)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
    ws = pa.prefill_workspace(plan)
    q, k, v = batch.q.cuda(), batch.k.cuda(), batch.v.cuda()
    outs, caches = [], []
    for _ in range(3):
        out = torch.full_like(q, float("nan"))
        pa.pa_prefill_varlen_int8_fused(dims, q, k, v, *gpu, plan, batch.scale, out, ws)
        outs.append(out)
        caches.append(tuple(t.clone() for t in gpu))
    torch.cuda.synchronize()
    for out, cache in zip(outs[1:], caches[1:]):
        assert torch.equal(out, outs[0])
        for a, b in zip(cache, caches[0]):
            assert torch.equal(a, b)
    assert pa.pa_read_device_error() == 0


def test_int8_fused_prefill_bad_slot_flagged():
    """A slot outside [-1, num_slots) is skipped and flagged (bit 0); -1 skips silently; every other
    row's codes and scales are stored exactly as pa_store_kvcache_int8 stores them."""
    w = workloads.random_case(831, num_seqs=2, hq=4, hkv=2, d=128, bs=16, max_len=200, cached=None, device="cuda")
    batch = w.batches[0]
    dims = dims_of(w, batch)
    gpu, _ = int8_pools(w, batch.num_heads)
    before = tuple(t.clone() for t in gpu)
    ref = tuple(t.clone() for t in gpu)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
    slots = plan.dev[plan.meta.off_slot_mapping:plan.meta.off_slot_mapping + 4 * batch.num_tokens].view(torch.int32)
    num_slots = w.pool.num_blocks * w.pool.block_size
    orig = slots.clone()
    slots[3] = num_slots + 5
    slots[7] = -1
    q, k, v = batch.q.cuda(), batch.k.cuda(), batch.v.cuda()
    out = torch.empty_like(q)
    pa.pa_prefill_varlen_int8_fused(dims, q, k, v, *gpu, plan, batch.scale, out)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() & 1
    # the store kernel on the same slots (3 and 7 skipped there too) gives the same cache
    pa.pa_store_kvcache_int8(dims, k, v, *ref, slots, batch.num_tokens)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() & 1
    for a, b in zip(gpu, ref):
        assert torch.equal(a, b)
    hkv, d = w.pool.num_kv_heads, w.pool.head_dim
    codes, codes0 = gpu[0].view(num_slots, hkv, d), before[0].view(num_slots, hkv, d)
    for t in (3, 7):
        s = int(orig[t])
        assert torch.equal(codes[s], codes0[s]), f"row {t} was written"


def test_int8_fused_prefill_two_plans_on_two_streams():
    """Two batches with plans and workspaces of their own, launched on two streams without ordering
    between them: both give the oracle's result."""
    ws = [workloads.random_case(seed, num_seqs=24, hq=8, hkv=2, d=128, bs=16, max_len=600, cached="random",
                                device="cuda") for seed in (841, 842)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    runs = []
    for w, st in zip(ws, streams):
        batch = w.batches[0]
        gpu, host = int8_pools(w, batch.num_heads)
        dims = dims_of(w, batch)
        q, k, v = batch.q.cuda(), batch.k.cuda(), batch.v.cuda()
        plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
        out = torch.full_like(q, float("nan"))
        runs.append((w, batch, gpu, host, dims, q, k, v, plan, out, st))
    torch.cuda.synchronize()
    for w, batch, gpu, host, dims, q, k, v, plan, out, st in runs:
        pa.pa_prefill_varlen_int8_fused(dims, q, k, v, *gpu, plan, batch.scale, out, stream=st)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    for w, batch, gpu, host, dims, q, k, v, plan, out, st in runs:
        ref, _ = oracle.run_batch_int8(*host, batch, w.pool.block_size)
        int8_equal(gpu, host, what=f"{w.name} (two streams)")
        assert_close(out, ref, what=f"int8 fused on its own stream ({w.name})")
