"""INT8 KV cache on the GPU: quantising store bit-exact against the oracle,
fused-dequant decode within tolerance of the oracle's attention over the
dequantised cache.

Source of the method: "面试问答准备: nano-vLLM 推理引擎优化", Q3 (KV cache
quantisation to int8 with per-token, per-head scales).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import (assert_close, int8_equal, int8_pools, run_gpu_decode_int8)

pytestmark = pytest.mark.gpu


def _special_rows(t, hkv, d, seed):
    """Random N(0, 1) rows plus rows that exercise the rounding rule's corners."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(t, hkv, d, generator=g)
    x[0] = 0.0                                   # all-zero vector: scale floored at 1e-8, codes 0
    x[1] = 1e-20 * torch.randn(hkv, d, generator=g)  # below the floor: scale 1e-8 exactly, codes 0
    x[2] = torch.randn(hkv, d, generator=g) * 1e4
    x[3, :, 0] = 127.0                           # scale = 1.0: every other value quantised as itself
    x[3, :, 1:] = torch.tensor([2.5, -3.5, 0.5, -0.5, 126.5, -126.5, 64.25, -1.0])[torch.arange(d - 1) % 8]
    x[4, :, 0] = -254.0                          # negative extreme sets the scale (2.0)
    x[5] = torch.where(torch.arange(d) % 2 == 0, torch.tensor(1e-3), torch.tensor(-3e38))[None]  # near bf16 max
    # the scale stored as fp16 leaves the normal range: max|x| ~ 6e-6 (< 1e-5) gives a scale of
    # a few fp16 subnormal steps, max|x| ~ 3e-3 one with a few bits (both sides must agree)
    x[6] = 2e-6 * torch.randn(hkv, d, generator=g)
    x[7] = 1e-3 * torch.randn(hkv, d, generator=g)
    # max|x| = a with a/127 inexact in fp32 and x = +-a/2: x/scale lies within an ulp of 63.5, so
    # the IEEE quotient alone decides between codes 63 and 64 (for bf16 inputs the only
    # half-integer quotients besides those of power-of-two scales).  For these four a, x times
    # the rounded reciprocal of the scale lands on the other side of 63.5 (9, 13: quotient
    # 63.499996, code 63; 15, 19: quotient 63.5, code 64)
    for row, a in zip(range(8, 12), (9.0, 13.0 * 2 ** -7, 15.0 * 2 ** 5, 19.0 * 2 ** -20)):
        x[row] = torch.where(torch.arange(d) % 2 == 0, torch.tensor(a / 2), torch.tensor(-a / 2))[None]
        x[row, :, 0] = a
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_store_int8_bit_exact(d):
    """Codes and fp16 scales equal the oracle's bit for bit; -1 slots write nothing."""
    nb, bs, hkv, hq, t = 9, 16, 3, 6, 120
    g = torch.Generator().manual_seed(300 + d)
    slots = torch.randperm(nb * bs, generator=g)[:t].to(torch.int32)
    slots[torch.randperm(t, generator=g)[:17]] = -1
    k, v = _special_rows(t, hkv, d, 1 + d), _special_rows(t, hkv, d, 2 + d)
    dims = pa.make_dims(nb, bs, hq, hkv, d)
    gpu = pa.int8_cache(dims, "cuda")
    pa.pa_store_kvcache_int8(dims, k.cuda(), v.cuda(), *gpu, slots.cuda(), t)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    host = (np.zeros((nb, bs, hkv, d), np.int8), np.zeros((nb, bs, hkv, d), np.int8),
            np.zeros((nb, hkv, bs), np.uint16), np.zeros((nb, hkv, bs), np.uint16))
    oracle.store_kvcache_int8(*host, k, v, slots.numpy())
    int8_equal(gpu, host, what=f"store d={d}")
    # the corner rows came out as the rounding rule says (checked on the GPU result directly)
    kc = gpu[0].cpu().numpy().reshape(nb * bs, hkv, d)
    s3 = int(slots[3])
    if s3 >= 0:
        row = kc[s3, 0]
        assert row[0] == 127 and list(row[1:7]) == [3, -4, 1, -1, 127, -127]


def test_store_int8_bad_slot_flagged():
    nb, bs, hkv, d = 4, 16, 1, 64
    dims = pa.make_dims(nb, bs, 2, hkv, d)
    gpu = pa.int8_cache(dims, "cuda")
    k = torch.randn(3, hkv, d, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([0, nb * bs, -1], dtype=torch.int32, device="cuda")
    pa.pa_store_kvcache_int8(dims, k, k, *gpu, slots, 3)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() & 1
    assert int(gpu[0].view(-1, hkv * d)[1:].abs().sum()) == 0  # nothing but slot 0 written


def test_pool_quantise_bit_exact_qwen3_pool():
    """The whole Qwen3-8B decode pool (~1,200 blocks of 256 tokens) quantised on both sides."""
    w = workloads.make("qwen3_decode", device="cuda")
    gpu, host = int8_pools(w, w.batches[0].num_heads)
    int8_equal(gpu, host, what="qwen3 pool")


def _decode_case(w, split):
    batch = w.batches[-1]
    gpu, host = int8_pools(w, batch.num_heads)
    out, plan = run_gpu_decode_int8(w, batch, gpu, split_tokens=split)
    ref, _ = oracle.run_batch_int8(*host, batch, w.pool.block_size)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(gpu, host, what="cache after the decode step's store")
    return out, ref, plan


@pytest.mark.parametrize("split", [0, 64, 256])
def test_decode_int8_qwen3(split):
    out, ref, plan = _decode_case(workloads.make("qwen3_decode", device="cuda"), split)
    if split:
        assert plan.meta.max_splits > 1
    assert_close(out, ref, what=f"int8 qwen3 decode split={split}")


CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len
    (401, 5, 2, 1, 64, 16, 300),
    (402, 7, 4, 2, 64, 256, 900),
    (403, 9, 7, 1, 128, 16, 700),
    (404, 4, 16, 1, 128, 32, 500),
    (405, 6, 8, 8, 128, 1024, 2100),
    (406, 3, 28, 4, 128, 16, 1500),
    (407, 8, 12, 1, 64, 64, 200),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
@pytest.mark.parametrize("split", [0, 64])
def test_decode_int8_random(case, split):
    seed, B, hq, hkv, d, bs, max_len = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, kind="decode",
                              device="cuda")
    out, ref, _ = _decode_case(w, split)
    assert_close(out, ref, what=f"int8 case {seed} split {split}")


def test_decode_int8_short_contexts():
    """Contexts 1..20 tokens: single partial chunks, tails inside the first chunk."""
    w = workloads.random_case(411, num_seqs=20, hq=8, hkv=2, d=128, bs=16, min_len=20, max_len=20,
                              kind="decode", device="cuda")
    w.batches[0].seq_lens[:] = np.arange(1, 21, dtype=np.int32)
    out, ref, _ = _decode_case(w, 0)
    assert_close(out, ref, what="int8 short contexts")


def test_decode_int8_deterministic():
    w = workloads.random_case(412, num_seqs=6, hq=16, hkv=2, d=128, bs=16, max_len=3000, kind="decode",
                              device="cuda")
    batch = w.batches[0]
    gpu, _ = int8_pools(w, batch.num_heads)
    a, _ = run_gpu_decode_int8(w, batch, gpu, split_tokens=256)
    b, _ = run_gpu_decode_int8(w, batch, gpu, split_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("case", [(421, 7, 8, 2, 128, 16, 900), (422, 5, 12, 1, 64, 32, 700),
                                  (423, 6, 16, 1, 128, 256, 1500)], ids=["421", "422", "423"])
@pytest.mark.parametrize("split", [0, 64])
def test_decode_int8_fused(case, split):
    """Quantising store + INT8 decode in one launch: cache bit-exact, output as the oracle's."""
    seed, B, hq, hkv, d, bs, max_len = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, kind="decode",
                              device="cuda")
    batch = w.batches[0]
    gpu, host = int8_pools(w, batch.num_heads)
    dims = pa.make_dims(w.pool.num_blocks, w.pool.block_size, batch.num_heads, w.pool.num_kv_heads,
                        w.pool.head_dim)
    plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split).upload("cuda")
    ws = pa.decode_workspace(plan)
    out = torch.empty_like(batch.q)
    pa.pa_decode_int8_fused(dims, batch.q, batch.k, batch.v, *gpu, plan, batch.scale, out, ws)
    ref, _ = oracle.run_batch_int8(*host, batch, w.pool.block_size)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(gpu, host, what="cache after the fused store")
    assert_close(out, ref, what=f"int8 fused case {seed} split {split}")
    # and the unfused pair on the same (now stored) cache agrees up to rounding order
    out2 = torch.empty_like(batch.q)
    pa.pa_decode_int8(dims, batch.q, *gpu, plan, batch.scale, out2, ws)
    torch.cuda.synchronize()
    assert (out.float() - out2.float()).abs().max().item() < 1e-2
