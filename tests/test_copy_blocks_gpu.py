"""Block copy (copy-on-write fork) parity: the whole cache byte-identical to the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from tests.harness import bits, int8_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs,hkv,d", [(16, 4, 128), (256, 8, 128), (32, 1, 64)])
def test_copy_blocks_bit_exact(bs, hkv, d):
    g = torch.Generator(device="cuda").manual_seed(bs + hkv)
    nb = 40
    kc = torch.randn(nb, bs, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(bs)
    blocks = rng.permutation(nb)
    srcs, dsts = blocks[:10], blocks[10:20]  # disjoint
    ns = rng.integers(0, bs + 1, size=10)
    ns[0], ns[1] = bs, 1
    triples = np.stack([srcs, dsts, ns], 1).astype(np.int32)
    want_k, want_v = bits(kc), bits(vc)
    oracle.copy_blocks(want_k, want_v, triples, bs)
    dims = pa.make_dims(nb, bs, hkv * 2, hkv, d)
    pa.pa_copy_blocks(dims, kc, vc, torch.from_numpy(triples).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), want_k) and np.array_equal(bits(vc), want_v)
    assert pa.pa_read_device_error() == 0


def test_copy_blocks_rejects_out_of_range_triples():
    nb, bs = 4, 16
    kc = torch.zeros(nb, bs, 1, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    before = bits(kc)
    dims = pa.make_dims(nb, bs, 1, 1, 64)
    bad = torch.tensor([[0, nb, 3], [1, 2, bs + 1]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(dims, kc, vc, bad)
    assert pa.pa_read_device_error() & 4
    assert np.array_equal(bits(kc), before)


@pytest.mark.parametrize("bs,hkv,d", [(16, 4, 128), (256, 8, 128), (32, 1, 64)])
def test_copy_blocks_int8_bit_exact(bs, hkv, d):
    """INT8 cache fork: codes and every head's scale run byte-identical to the oracle's copy."""
    g = torch.Generator(device="cuda").manual_seed(bs + hkv + 1)
    nb = 40
    dims = pa.make_dims(nb, bs, hkv * 2, hkv, d)
    n = nb * bs
    cache = pa.int8_cache(dims, "cuda")
    k = torch.randn(n, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(n, hkv, d, device="cuda", generator=g).to(torch.bfloat16)
    pa.pa_store_kvcache_int8(dims, k, v, *cache, torch.arange(n, dtype=torch.int32, device="cuda"), n)
    torch.cuda.synchronize()
    host = [c.cpu().numpy() for c in cache]
    host = [h.view(np.uint16) if h.dtype == np.float16 else h.copy() for h in host]
    rng = np.random.default_rng(bs + 1)
    blocks = rng.permutation(nb)
    srcs, dsts = blocks[:10], blocks[10:20]
    ns = rng.integers(0, bs + 1, size=10)
    ns[0], ns[1] = bs, 1
    triples = np.stack([srcs, dsts, ns], 1).astype(np.int32)
    oracle.copy_blocks_int8(*host, triples)
    pa.pa_copy_blocks_int8(dims, *cache, torch.from_numpy(triples).cuda())
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(cache, host, what=f"int8 copy bs={bs}")
