"""Decode parity against the fp64 oracle, split-KV consistency and decode == last prefill row."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, bits, dims_of, run_gpu_batch

pytestmark = pytest.mark.gpu


def _run(w, split_tokens=0):
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    res = []
    for batch in w.batches:
        out, plan = run_gpu_batch(w, batch, kc, vc, split_tokens=split_tokens)
        ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size)
        res.append((batch, out, ref, plan))
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    return res


def test_decode_tiny_after_prefill():
    """Tiny case: store + prefill both prompts, then one decode step per sequence."""
    res = _run(workloads.tiny(device="cuda"))
    for batch, out, ref, _ in res:
        assert_close(out, ref, what=batch.kind)


@pytest.mark.parametrize("split", [0, 64, 256])
def test_decode_qwen3(split):
    (batch, out, ref, plan), = _run(workloads.make("qwen3_decode", device="cuda"), split_tokens=split)
    if split:
        assert plan.meta.max_splits > 1
    assert_close(out, ref, what=f"qwen3 decode split={split}")


CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len
    (201, 5, 2, 1, 64, 16, 300),
    (202, 7, 4, 2, 64, 256, 900),
    (203, 9, 7, 1, 128, 16, 700),
    (204, 4, 16, 1, 128, 32, 500),
    (205, 6, 8, 8, 128, 1024, 2100),
    (206, 3, 28, 4, 128, 16, 1500),
    (207, 8, 12, 1, 64, 64, 200),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
@pytest.mark.parametrize("split", [0, 64])
def test_decode_random(case, split):
    seed, B, hq, hkv, d, bs, max_len = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, kind="decode",
                              device="cuda")
    (batch, out, ref, _), = _run(w, split)
    assert_close(out, ref, what=f"case {seed} split {split}")


def test_split_counts_agree():
    """S = 1 against S = 2, 4, 16 on the same inputs: the LSE combine reproduces one pass."""
    w = workloads.random_case(211, num_seqs=4, hq=8, hkv=2, d=128, bs=16, max_len=4096, min_len=4096,
                              kind="decode", device="cuda")
    outs = {}
    for split in (4096, 2048, 1024, 256):
        (batch, out, ref, plan), = _run(w, split)
        outs[plan.meta.max_splits] = out.double().cpu().numpy()
    base = outs[1]
    for s, o in outs.items():
        rel = np.abs(o - base).max() / np.abs(base).max()
        assert rel < 1e-2, (s, rel)


def test_decode_equals_last_prefill_row_on_gpu():
    """Decode at context n equals row n-1 of a full prefill over the same n tokens."""
    n, hq, hkv, d, bs = 777, 14, 2, 128, 16
    g = torch.Generator(device="cuda").manual_seed(12)
    mk = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)
    nb = -(-n // bs) + 3
    blocks = [np.random.default_rng(3).permutation(nb)[:-(-n // bs)].astype(np.int32)]
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    q, k, v = mk(n, hq, d), mk(n, hkv, d), mk(n, hkv, d)
    full = workloads.Batch("prefill", np.array([n], np.int32), np.array([n], np.int32), blocks, q, k, v, hq, d ** -0.5)
    w = workloads.Workload("x", pool, [])
    kc, vc = pool.k_cache.clone(), pool.v_cache.clone()
    out_full, _ = run_gpu_batch(w, full, kc, vc)
    dec = workloads.Batch("decode", np.array([n], np.int32), np.array([1], np.int32), blocks,
                          q[n - 1:].contiguous(), k[n - 1:].contiguous(), v[n - 1:].contiguous(), hq, d ** -0.5)
    for split in (0, 64):
        out_dec, _ = run_gpu_batch(w, dec, kc, vc, split_tokens=split)
        torch.cuda.synchronize()
        assert_close(out_dec, out_full[n - 1:].double().cpu().numpy(), what=f"decode vs prefill split={split}")


def test_decode_zero_context_writes_zeros():
    dims = pa.make_dims(4, 16, 4, 2, 64)
    plan = pa.pa_pack_decode(dims, [0, 3], [[], [1]]).upload()
    g = torch.Generator(device="cuda").manual_seed(2)
    kc = torch.randn(4, 16, 2, 64, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(2, 4, 64, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.full_like(q, 7.0)
    pa.pa_decode(dims, q, kc, kc, plan, 0.125, out, pa.decode_workspace(plan))
    torch.cuda.synchronize()
    assert (out[0] == 0).all()
    assert torch.isfinite(out[1].float()).all() and not (out[1] == 7.0).any()


def test_decode_qwen25_full_size_every_sequence():
    """64 x 32768, Hq 28 / Hkv 4, block 16, fully permuted (the benched decode batch): the full
    launch against the oracle on all 64 sequences."""
    w = workloads.make("qwen25_decode", device="cuda")
    batch = w.batches[0]
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    kc, vc = w.pool.k_cache, w.pool.v_cache  # modified in place by the store
    out, plan = run_gpu_batch(w, batch, kc, vc)
    torch.cuda.synchronize()
    assert plan.meta.max_splits > 1
    assert pa.pa_read_device_error() == 0
    ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size)
    assert_close(out, ref, what="qwen25 decode (every sequence)")


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_two_split_plans_share_an_uninitialised_workspace(kv):
    """Plans with different split counts on one workspace holding junk: both match the
    oracle, and the same plan run again gives the same bits."""
    from tests.harness import int8_pools
    w = workloads.random_case(151, num_seqs=6, hq=8, hkv=2, d=128, bs=16, max_len=2000, kind="decode",
                              device="cuda")
    b = w.batches[0]
    dims = dims_of(w, b)
    plans = [pa.pa_pack_decode(dims, b.seq_lens, b.block_lists, s).upload("cuda") for s in (256, 576)]
    assert plans[0].meta.max_splits > plans[1].meta.max_splits > 1
    ws = torch.full((max(int(p.meta.workspace_bytes) for p in plans),), 0x5A, dtype=torch.uint8, device="cuda")
    q, k, v = b.q.cuda(), b.k.cuda(), b.v.cuda()
    if kv == "bf16":
        kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
        pa.pa_store_kvcache(dims, k, v, kc, vc, plans[0].slot_mapping, b.num_tokens)
        ref, _ = oracle.run_batch(bits(w.pool.k_cache), bits(w.pool.v_cache), b, w.pool.block_size)
        call = lambda p, out: pa.pa_decode(dims, q, kc, vc, p, b.scale, out, ws)
    else:
        gpu, host = int8_pools(w, b.num_heads)
        pa.pa_store_kvcache_int8(dims, k, v, *gpu, plans[0].slot_mapping, b.num_tokens)
        ref, _ = oracle.run_batch_int8(*host, b, w.pool.block_size)  # stores the batch's rows, then attends
        call = lambda p, out: pa.pa_decode_int8(dims, q, *gpu, p, b.scale, out, ws)
    outs = []
    for rep in range(2):
        for p in plans:
            out = torch.empty_like(q)
            call(p, out)
            outs.append(out)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    for out in outs:
        assert_close(out, ref, what=f"{kv} shared workspace")
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[3])
