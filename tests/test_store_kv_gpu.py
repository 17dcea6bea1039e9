"""KV scatter parity: the whole cache must be byte-identical to the oracle's scatter."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import bits, dims_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefill_256", "qwen3_prefix", "qwen3_chunked", "qwen3_decode",
                                  "qwen25_prefill"])
def test_store_matches_oracle_bit_exact(name):
    w = workloads.make(name, device="cuda")
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    for batch in w.batches:
        dims = dims_of(w, batch)
        if batch.kind == "prefill":
            plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload()
        else:
            plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists).upload()
        pa.pa_store_kvcache(dims, batch.k, batch.v, kc, vc, plan.slot_mapping, batch.num_tokens)
        slots = oracle.slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, w.pool.block_size)
        oracle.store_kvcache(ok_, ov_, batch.k, batch.v, slots)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), ok_)
    assert np.array_equal(bits(vc), ov_)
    assert pa.pa_read_device_error() == 0


def test_store_skips_padding_and_rejects_out_of_range_slots():
    g = torch.Generator(device="cuda").manual_seed(3)
    nb, bs, hkv, d, t = 6, 16, 2, 64, 40
    kc = torch.randn(nb, bs, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(t, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(t, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(4))[:t].to(torch.int32)
    slots[::5] = -1  # CUDA-graph padding tokens
    want_k, want_v = bits(kc), bits(vc)
    oracle.store_kvcache(want_k, want_v, k, v, slots.numpy())
    dims = pa.make_dims(nb, bs, 4, hkv, d)
    pa.pa_store_kvcache(dims, k, v, kc, vc, slots.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), want_k) and np.array_equal(bits(vc), want_v)
    assert pa.pa_read_device_error() == 0
    # a slot past the pool is skipped by the kernel's bounds check and reported
    bad = slots.clone()
    bad[1] = nb * bs + 7
    before = bits(kc)
    pa.pa_store_kvcache(dims, k, v, kc, vc, bad.cuda())
    assert pa.pa_read_device_error() & 1
    assert pa.pa_read_device_error() == 0  # reading clears it
    after = bits(kc)
    # every other token landed (same bytes as before, the store is idempotent), nothing else changed
    assert np.array_equal(after, before)
