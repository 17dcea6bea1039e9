"""Fused store + decode, and decode replayed from a CUDA graph over a fixed-shape plan.

Sources: "手搓 vLLM 推理引擎", Step 4 (store the new K/V, then attend over the
cache including them) and Step 5 (decode captured as a CUDA graph per
batch-size bucket; unused rows get slot -1 and context length 0).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, bits, dims_of

pytestmark = pytest.mark.gpu


def _fused_vs_oracle(w, split):
    batch = w.batches[-1]
    dims = dims_of(w, batch)
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(kc), bits(vc)
    plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split).upload("cuda")
    ws = pa.decode_workspace(plan)
    out = torch.empty_like(batch.q)
    pa.pa_decode_fused(dims, batch.q, batch.k, batch.v, kc, vc, plan, batch.scale, out, ws)
    ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    # the fused store wrote exactly what the oracle's store wrote
    assert np.array_equal(bits(kc), ok_) and np.array_equal(bits(vc), ov_)
    # and attention equals the unfused pair (store, then decode) up to rounding order
    kc2, vc2 = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    out2 = torch.empty_like(batch.q)
    pa.pa_store_kvcache(dims, batch.k, batch.v, kc2, vc2, plan.slot_mapping, batch.num_tokens)
    pa.pa_decode(dims, batch.q, kc2, vc2, plan, batch.scale, out2, ws)
    torch.cuda.synchronize()
    assert (out.float() - out2.float()).abs().max().item() < 1e-2
    return out, ref


@pytest.mark.parametrize("split", [0, 64, 256])
def test_fused_decode_qwen3(split):
    out, ref = _fused_vs_oracle(workloads.make("qwen3_decode", device="cuda"), split)
    assert_close(out, ref, what=f"fused qwen3 decode split={split}")


CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len
    (601, 5, 2, 1, 64, 16, 300),
    (602, 9, 7, 1, 128, 16, 700),
    (603, 4, 16, 1, 128, 32, 500),
    (604, 3, 28, 4, 128, 16, 1500),
    (605, 8, 12, 1, 64, 64, 200),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
@pytest.mark.parametrize("split", [0, 64])
def test_fused_decode_random(case, split):
    seed, B, hq, hkv, d, bs, max_len = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, kind="decode",
                              device="cuda")
    out, ref = _fused_vs_oracle(w, split)
    assert_close(out, ref, what=f"fused case {seed} split {split}")


def _bucket_step(rng, B, real, max_ctx, nb, bs, hq, hkv, d, gen):
    """One decode step of a bucket: `real` live sequences, B - real padding entries (context 0)."""
    ctx = np.zeros(B, np.int32)
    ctx[:real] = rng.integers(1, max_ctx + 1, real)
    perm = rng.permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for c in ctx:
        n = -(-int(c) // bs)
        blocks.append(perm[o:o + n])
        o += n
    mk = lambda *s: torch.randn(*s, device="cuda", generator=gen).to(torch.bfloat16)
    return ctx, blocks, mk(B, hq, d), mk(B, hkv, d), mk(B, hkv, d)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("d,hq,hkv,split", [(128, 16, 2, 256), (64, 12, 1, 64), (128, 28, 4, 0)])
def test_decode_graph_replay_fixed_bucket(kv, fused, d, hq, hkv, split):
    """Capture once, replay on three steps with new contexts, blocks and padding."""
    B, max_ctx, bs = 8, 1024, 16
    nb = B * (max_ctx // bs) + 4
    rng = np.random.default_rng(700 + d + hq)
    gen = torch.Generator(device="cuda").manual_seed(701)
    kc = torch.randn(nb, bs, hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
    dims = pa.make_dims(nb, bs, hq, hkv, d)
    scale = d ** -0.5
    ctx, blocks, q, k, v = _bucket_step(rng, B, 5, max_ctx, nb, bs, hq, hkv, d, gen)
    plan = pa.pa_pack_decode_fixed(dims, ctx, blocks, max_ctx, split).upload("cuda")
    ws = pa.decode_workspace(plan)
    q_in, k_in, v_in = q.clone(), k.clone(), v.clone()  # the graph's input buffers
    out = torch.zeros(B, hq, d, dtype=torch.bfloat16, device="cuda")
    shape = tuple(getattr(plan.meta, f) for f in ("num_items", "total_bytes", "workspace_bytes", "off_items"))

    if kv == "int8":  # the pool quantised slot by slot; the caches below are what the graph reads and writes
        c8 = pa.int8_cache(dims, "cuda")
        n_slots = nb * bs
        pa.pa_store_kvcache_int8(dims, kc.view(n_slots, hkv, d), vc.view(n_slots, hkv, d), *c8,
                                 torch.arange(n_slots, dtype=torch.int32, device="cuda"), n_slots)

    def step():
        if kv == "int8" and fused:
            pa.pa_decode_int8_fused(dims, q_in, k_in, v_in, *c8, plan, scale, out, ws)
        elif kv == "int8":
            pa.pa_store_kvcache_int8(dims, k_in, v_in, *c8, plan.slot_mapping, B)
            pa.pa_decode_int8(dims, q_in, *c8, plan, scale, out, ws)
        elif fused:
            pa.pa_decode_fused(dims, q_in, k_in, v_in, kc, vc, plan, scale, out, ws)
        else:
            pa.pa_store_kvcache(dims, k_in, v_in, kc, vc, plan.slot_mapping, B)
            pa.pa_decode(dims, q_in, kc, vc, plan, scale, out, ws)

    def host_cache():
        if kv == "int8":
            h = [c.cpu().numpy() for c in c8]
            return [x.view(np.uint16) if x.dtype == np.float16 else x.copy() for x in h]
        return [bits(kc), bits(vc)]

    step()  # first call outside capture: one-time set-up (function attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for it, real in enumerate((5, 8, 1)):
        if it > 0:
            ctx, blocks, q, k, v = _bucket_step(rng, B, real, max_ctx, nb, bs, hq, hkv, d, gen)
            pa.pa_pack_decode_fixed(dims, ctx, blocks, max_ctx, split, into=plan)
            assert tuple(getattr(plan.meta, f) for f in ("num_items", "total_bytes", "workspace_bytes",
                                                         "off_items")) == shape
            plan.upload("cuda")  # same device buffer the graph reads
            q_in.copy_(q), k_in.copy_(k), v_in.copy_(v)
        torch.cuda.synchronize()
        before = host_cache()
        out.fill_(1.0)
        graph.replay()
        torch.cuda.synchronize()
        assert pa.pa_read_device_error() == 0
        live = workloads.Batch("decode", ctx[:real], np.ones(real, np.int32), blocks[:real], q[:real].cpu(),
                               k[:real].cpu(), v[:real].cpu(), hq, scale)
        if kv == "int8":
            ref, _ = oracle.run_batch_int8(*before, live, bs)
        else:
            ref, _ = oracle.run_batch(*before, live, bs)
        assert_close(out[:real], ref, what=f"graph step {it} kv={kv} fused={fused} d={d} real={real}")
        assert not out[real:].float().abs().any(), "padding rows must be zero"
        for got, want in zip(host_cache(), before):
            assert np.array_equal(got, want), "cache after the step"
