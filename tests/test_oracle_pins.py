"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: hand-worked
fixtures, a pure-Python brute force, closed forms, invariants and a library
routine (torch's fp64 attention on the CPU).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from paged_kv_cache_kvcache_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _f64(t):
    return t.to(torch.float64).numpy()


def _identity_case(seed, num_seqs, hq, hkv, d, bs, max_len, cached=True):
    """Blocks of sequence b are consecutive (identity layout), so the dense
    keys of b are a plain slice of the pool: no slot arithmetic needed."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (num_seqs,), generator=g).numpy().astype(np.int32)
    if cached:
        qlens = np.array([int(torch.randint(1, int(l) + 1, (1,), generator=g)) for l in lens], np.int32)
    else:
        qlens = lens.copy()
    nblk = [-(-int(l) // bs) for l in lens]
    starts = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int32)
    blocks = [np.arange(starts[b], starts[b + 1], dtype=np.int32) for b in range(num_seqs)]
    nb = int(starts[-1]) + 2
    pool_k = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    pool_v = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    t = int(qlens.sum())
    q = torch.randn(t, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(t, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(t, hkv, d, generator=g).to(torch.bfloat16)
    return dict(lens=lens, qlens=qlens, blocks=blocks, starts=starts, pool_k=pool_k, pool_v=pool_v,
                q=q, k=k, v=v, bs=bs, scale=1.0 / np.sqrt(d))


def _contiguous_kv(c, b):
    """Dense K/V of sequence b for the identity layout: cached prefix is a
    slice of the pool, the new tokens follow."""
    bs = c["bs"]
    lk, lq = int(c["lens"][b]), int(c["qlens"][b])
    t0 = int(c["qlens"][:b].sum())
    hkv, d = c["pool_k"].shape[2], c["pool_k"].shape[3]
    flat_k = c["pool_k"].reshape(-1, hkv, d)
    flat_v = c["pool_v"].reshape(-1, hkv, d)
    s0 = int(c["starts"][b]) * bs
    kk = torch.cat([flat_k[s0:s0 + lk - lq], c["k"][t0:t0 + lq]])
    vv = torch.cat([flat_v[s0:s0 + lk - lq], c["v"][t0:t0 + lq]])
    return kk, vv


def _oracle_case(c):
    pk, pv = _bits(c["pool_k"]), _bits(c["pool_v"])
    slots = oracle.slot_mapping(c["lens"], c["qlens"], c["blocks"], c["bs"])
    oracle.store_kvcache(pk, pv, c["k"], c["v"], slots)
    out, pairs = oracle.paged_attention(c["q"], pk, pv, c["lens"], c["qlens"], c["blocks"], c["bs"], c["scale"])
    return out, pairs, pk, pv


# ---------------------------------------------------------------- fixtures


def test_gather_golden():
    fx = json.load(open(os.path.join(GOLDEN, "gather_toy.json")))
    pool = torch.tensor(fx["pool"], dtype=torch.float32).to(torch.bfloat16)
    for s in fx["sequences"]:
        dense = oracle.gather_dense(pool, s["len"], s["blocks"], fx["block_size"])
        assert dense.tolist() == [[[float(x) for x in h] for h in row] for row in s["expected"]]


def test_slot_mapping_golden():
    fx = json.load(open(os.path.join(GOLDEN, "slot_mapping_toy.json")))
    seqs = fx["sequences"]
    lens = [s["len"] for s in seqs]
    qlens = [s["len"] - s["num_cached"] for s in seqs]
    blocks = [s["blocks"] for s in seqs]
    got = oracle.slot_mapping(lens, qlens, blocks, fx["block_size"])
    want = sum((s["expected_slots"] for s in seqs), [])
    assert got.tolist() == want


def test_slot_mapping_rejects_short_block_list():
    with pytest.raises(ValueError):
        oracle.slot_mapping([17], [17], [[0]], 16)


# ---------------------------------------------------------------- scatter


def test_scatter_matches_fancy_index_and_keeps_canary():
    g = torch.Generator().manual_seed(11)
    nb, bs, hkv, d, t = 9, 4, 3, 8, 13
    kc = _bits(torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16))
    vc = _bits(torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16))
    k = torch.randn(t, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(t, hkv, d, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:t].numpy().astype(np.int32)
    slots[[2, 7]] = -1  # padded tokens
    want_k, want_v = kc.copy(), vc.copy()
    ok = slots >= 0
    want_k.reshape(nb * bs, -1)[slots[ok]] = _bits(k).reshape(t, -1)[ok]
    want_v.reshape(nb * bs, -1)[slots[ok]] = _bits(v).reshape(t, -1)[ok]
    before = kc.copy()
    oracle.store_kvcache(kc, vc, k, v, slots)
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)
    untouched = np.setdiff1d(np.arange(nb * bs), slots[ok])
    assert np.array_equal(kc.reshape(nb * bs, -1)[untouched], before.reshape(nb * bs, -1)[untouched])


# ---------------------------------------------------------------- attention vs brute force


@pytest.mark.parametrize("seed,hq,hkv,bs,cached", [(1, 4, 2, 4, True), (2, 3, 1, 5, False), (3, 2, 2, 8, True)])
def test_oracle_matches_brute_force(seed, hq, hkv, bs, cached):
    c = _identity_case(seed, num_seqs=3, hq=hq, hkv=hkv, d=16, bs=bs, max_len=24, cached=cached)
    out, _, _, _ = _oracle_case(c)
    t0 = 0
    for b in range(3):
        kk, vv = _contiguous_kv(c, b)
        lq = int(c["qlens"][b])
        qb = _f64(c["q"][t0:t0 + lq]).tolist()
        ref = np.array(brute.attention(qb, _f64(kk).tolist(), _f64(vv).tolist(), c["scale"]))
        np.testing.assert_allclose(out[t0:t0 + lq], ref, rtol=0, atol=1e-12)
        t0 += lq


def test_tiny_workload_matches_brute_force_on_numpy_gather():
    """Seeded tiny case (permuted pool): dense K/V rebuilt independently by
    numpy advanced indexing, pool[blocks[pos // bs], pos % bs]."""
    w = workloads.tiny()
    bs = w.pool.block_size
    pk, pv = _bits(w.pool.k_cache), _bits(w.pool.v_cache)
    for batch in w.batches:
        out, _ = oracle.run_batch(pk, pv, batch, bs)
        t0 = 0
        for b in range(batch.num_seqs):
            lk, lq = int(batch.seq_lens[b]), int(batch.query_lens[b])
            pos = np.arange(lk)
            blk = batch.block_lists[b][pos // bs]
            kk = torch.from_numpy(pk.view(np.int16)[blk, pos % bs].copy()).view(torch.bfloat16)
            vv = torch.from_numpy(pv.view(np.int16)[blk, pos % bs].copy()).view(torch.bfloat16)
            qb = _f64(batch.q[t0:t0 + lq]).tolist()
            ref = np.array(brute.attention(qb, _f64(kk).tolist(), _f64(vv).tolist(), batch.scale))
            np.testing.assert_allclose(out[t0:t0 + lq], ref, rtol=0, atol=1e-12)
            t0 += lq


def test_oracle_matches_torch_sdpa_fp64():
    """Library routine: torch CPU fp64 attention with a causal mask, Lq == Lk."""
    c = _identity_case(21, num_seqs=2, hq=6, hkv=2, d=32, bs=16, max_len=70, cached=False)
    out, _, _, _ = _oracle_case(c)
    t0 = 0
    for b in range(2):
        kk, vv = _contiguous_kv(c, b)
        lq = int(c["qlens"][b])
        q = c["q"][t0:t0 + lq].to(torch.float64).transpose(0, 1)
        k = kk.to(torch.float64).transpose(0, 1).repeat_interleave(3, dim=0)
        v = vv.to(torch.float64).transpose(0, 1).repeat_interleave(3, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=c["scale"])
        np.testing.assert_allclose(out[t0:t0 + lq], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        t0 += lq


# ---------------------------------------------------------------- invariants


def test_permutation_invariance_bit_exact():
    c = _identity_case(5, num_seqs=4, hq=4, hkv=2, d=16, bs=4, max_len=30, cached=True)
    out_a, _, _, _ = _oracle_case(c)
    nb = c["pool_k"].shape[0]
    sigma = torch.randperm(nb, generator=torch.Generator().manual_seed(99))
    inv = torch.empty_like(sigma)
    inv[sigma] = torch.arange(nb)
    c2 = dict(c)
    c2["pool_k"] = c["pool_k"][inv]  # new_pool[sigma[p]] = pool[p]
    c2["pool_v"] = c["pool_v"][inv]
    c2["blocks"] = [sigma.numpy()[b].astype(np.int32) for b in c["blocks"]]
    out_b, _, _, _ = _oracle_case(c2)
    assert np.array_equal(out_a, out_b)


def test_pair_count_closed_form():
    c = _identity_case(6, num_seqs=5, hq=3, hkv=1, d=8, bs=4, max_len=40, cached=True)
    _, pairs, _, _ = _oracle_case(c)
    lk, lq = c["lens"].astype(np.int64), c["qlens"].astype(np.int64)
    assert pairs == 3 * int(np.sum(lq * (lk - lq) + lq * (lq + 1) // 2))
    # full prefill of N tokens: N(N+1)/2 pairs per head
    n = 37
    c = _fixed_len_case(n, n, hq=1, hkv=1, d=8, bs=8, seed=7)
    _, pairs, _, _ = _oracle_case(c)
    assert pairs == n * (n + 1) // 2


def _fixed_len_case(lk, lq, hq, hkv, d, bs, seed, scale=None):
    g = torch.Generator().manual_seed(seed)
    nblk = -(-lk // bs)
    pool_k = torch.randn(nblk + 1, bs, hkv, d, generator=g).to(torch.bfloat16)
    pool_v = torch.randn(nblk + 1, bs, hkv, d, generator=g).to(torch.bfloat16)
    perm = torch.randperm(nblk + 1, generator=g).numpy().astype(np.int32)
    return dict(lens=np.array([lk], np.int32), qlens=np.array([lq], np.int32), blocks=[perm[:nblk]],
                starts=None, pool_k=pool_k, pool_v=pool_v,
                q=torch.randn(lq, hq, d, generator=g).to(torch.bfloat16),
                k=torch.randn(lq, hkv, d, generator=g).to(torch.bfloat16),
                v=torch.randn(lq, hkv, d, generator=g).to(torch.bfloat16),
                bs=bs, scale=scale if scale is not None else 1.0 / np.sqrt(d))


def test_prefix_suffix_equals_full_prefill_rows():
    """300-token sequence: querying only the last 44 (first 256 cached) gives
    exactly rows 256..299 of the full prefill."""
    full = _fixed_len_case(300, 300, hq=4, hkv=2, d=64, bs=256, seed=8)
    out_full, _, pk, pv = _oracle_case(full)
    out_sfx, _ = oracle.paged_attention(full["q"][256:], pk, pv, [300], [44], full["blocks"], 256, full["scale"])
    assert np.array_equal(out_sfx, out_full[256:])


def test_decode_equals_last_prefill_row():
    n = 65
    full = _fixed_len_case(n, n, hq=2, hkv=1, d=64, bs=16, seed=9)
    out_full, _, pk, pv = _oracle_case(full)
    out_dec, _ = oracle.paged_attention(full["q"][n - 1:], pk, pv, [n], [1], full["blocks"], 16, full["scale"])
    assert np.array_equal(out_dec[0], out_full[n - 1])


# ---------------------------------------------------------------- closed forms


def test_single_key_returns_its_value_exactly():
    c = _fixed_len_case(1, 1, hq=3, hkv=3, d=32, bs=16, seed=10)
    out, _, _, _ = _oracle_case(c)
    np.testing.assert_array_equal(out[0], _f64(c["v"][0]))


def test_zero_scale_gives_mean_of_visible_values():
    c = _fixed_len_case(20, 20, hq=2, hkv=1, d=16, bs=4, seed=12, scale=0.0)
    out, _, _, _ = _oracle_case(c)
    vv = _f64(c["v"])  # full prefill: the dense values are the new tokens' values
    for i in range(20):
        np.testing.assert_allclose(out[i, 0], vv[:i + 1, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_equal_keys_give_mean_of_values():
    c = _fixed_len_case(12, 12, hq=1, hkv=1, d=8, bs=4, seed=13)
    c["k"] = c["k"][:1].expand(12, 1, 8).contiguous()
    out, _, _, _ = _oracle_case(c)
    vv = _f64(c["v"])
    for i in range(12):
        np.testing.assert_allclose(out[i, 0], vv[:i + 1, 0].mean(axis=0), rtol=0, atol=1e-13)


def test_dominant_logit_selects_that_value():
    n, d, star = 10, 16, 6
    c = _fixed_len_case(n, n, hq=1, hkv=1, d=d, bs=4, seed=14, scale=1.0)
    k = torch.zeros(n, 1, d)
    for j in range(n):
        k[j, 0, j] = 1.0  # orthonormal keys
    c["k"] = k.to(torch.bfloat16)
    q = torch.zeros(n, 1, d)
    q[n - 1, 0, star] = 40.0
    c["q"] = q.to(torch.bfloat16)
    out, _, _, _ = _oracle_case(c)
    np.testing.assert_allclose(out[n - 1, 0], _f64(c["v"][star, 0]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- block copy (copy-on-write fork)


def test_copy_blocks_golden():
    fx = json.load(open(os.path.join(GOLDEN, "copy_blocks_toy.json")))
    k = _bits(torch.tensor(fx["k_pool"], dtype=torch.float32).to(torch.bfloat16))
    v = _bits(torch.tensor(fx["v_pool"], dtype=torch.float32).to(torch.bfloat16))
    oracle.copy_blocks(k, v, fx["triples"], fx["block_size"])
    want_k = _bits(torch.tensor(fx["expected_k"], dtype=torch.float32).to(torch.bfloat16))
    want_v = _bits(torch.tensor(fx["expected_v"], dtype=torch.float32).to(torch.bfloat16))
    assert np.array_equal(k, want_k) and np.array_equal(v, want_v)


def test_copy_blocks_matches_fancy_index():
    g = torch.Generator().manual_seed(31)
    nb, bs, hkv, d = 12, 16, 2, 8
    k = _bits(torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16))
    v = _bits(torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16))
    triples = np.array([[0, 5, 16], [3, 7, 9], [4, 11, 0], [1, 6, 1]], np.int32)
    want_k, want_v = k.copy(), v.copy()
    for s, t, n in triples:
        want_k[t, :n] = want_k[s, :n]
        want_v[t, :n] = want_v[s, :n]
    oracle.copy_blocks(k, v, triples, bs)
    assert np.array_equal(k, want_k) and np.array_equal(v, want_v)


def test_copy_blocks_int8_commutes_with_quantisation():
    """Forking a quantised cache equals quantising the forked bf16 cache: quantisation is per
    (token, KV head) and the fork moves whole tokens (a wrong scale index breaks this)."""
    g = torch.Generator().manual_seed(33)
    nb, bs, hkv, d = 10, 16, 3, 8
    pool_k = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    pool_v = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    triples = np.array([[0, 5, 16], [3, 7, 9], [4, 9, 0], [1, 6, 1], [2, 8, 15]], np.int32)

    def quantised(kb, vb):
        kc, ks = oracle.quantize_rows(kb)
        vc, vs = oracle.quantize_rows(vb)
        return (kc.copy(), vc.copy(), np.ascontiguousarray(ks.transpose(0, 2, 1)),
                np.ascontiguousarray(vs.transpose(0, 2, 1)))

    a = quantised(pool_k, pool_v)
    oracle.copy_blocks_int8(*a, triples)
    kb, vb = _bits(pool_k), _bits(pool_v)
    oracle.copy_blocks(kb, vb, triples, bs)
    b = quantised(torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16),
                  torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # and blocks outside every dst are untouched
    c = quantised(pool_k, pool_v)
    for x, y in zip(a, c):
        untouched = [blk for blk in range(nb) if blk not in triples[:, 1]]
        assert np.array_equal(x[untouched], y[untouched])


# ---------------------------------------------------------------- INT8 KV cache


def test_f16_conversion_matches_numpy():
    rng = np.random.default_rng(41)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-5).astype(np.float32),          # fp16 subnormals
        (rng.standard_normal(500) * 1e-8).astype(np.float32),           # rounds to +-0 or the smallest subnormal
        np.array([65504, 65519, 65520, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1e-8, 0.0, -0.0,
                  1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 1.0 / 127.0], dtype=np.float32),
    ])
    want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    back = np.array([oracle.f16_to_f32(int(h)) for h in want], dtype=np.float32)
    assert np.array_equal(back, want.view(np.float16).astype(np.float32))


def test_int8_quantize_golden():
    fx = json.load(open(os.path.join(GOLDEN, "int8_quant_toy.json")))
    for row in fx["rows"]:
        x = torch.tensor([row["x"]], dtype=torch.float32).to(torch.bfloat16)
        codes, scales = oracle.quantize_rows(x)
        assert codes[0].tolist() == row["codes"], row["note"]
        assert int(scales[0]) == row["scale_f16_bits"], row["note"]


def test_int8_quantize_invariants():
    g = torch.Generator().manual_seed(42)
    x = (torch.randn(500, 128, generator=g) * torch.rand(500, 1, generator=g) * 10).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1)
    # the largest element always maps to +-127 and nothing overflows
    assert np.abs(codes).max() <= 127
    assert (np.abs(codes).max(axis=1) == 127).all()
    # dequantised with the fp32 scale, every value is within half a step (plus the fp32
    # rounding of x / scale, which can move an exact ratio of k + 0.4999... onto k + 0.5)
    s32 = np.maximum(amax / np.float32(127.0), np.float32(1e-8)).astype(np.float32)
    err = np.abs(codes.astype(np.float64) * s32[:, None] - xf.astype(np.float64)) / s32[:, None]
    assert err.max() <= 0.5 + 1e-4
    # the stored scale is the fp16 rounding of that scale
    assert np.array_equal(scales, s32.astype(np.float16).view(np.uint16))


def test_int8_quantize_matches_fp32_formula_at_half_integer_quotients():
    """Rows whose quotient x / scale lies within an ulp of 63.5 (max|x| = a with a / 127 inexact in
    fp32, x = +-a/2): the code is decided by the IEEE fp32 quotient alone.  The oracle equals numpy's
    fp32 evaluation of the page's formula on them, and the product by the rounded reciprocal of the
    scale would give other codes on some (so these rows separate the two)."""
    rows = []
    for o in (9, 13, 15, 19, 33, 101):
        for j in (-20, -7, 0, 5):
            a = o * 2.0 ** j
            x = np.full(128, a / 2, np.float32)
            x[1::2] *= -1
            x[0] = a
            rows.append(x)
    x = torch.tensor(np.stack(rows)).to(torch.bfloat16)
    xf = x.float().numpy()
    assert np.array_equal(xf, np.stack(rows))  # every value exact in bf16
    codes, scales = oracle.quantize_rows(x)
    s = np.maximum(np.abs(xf).max(axis=1) / np.float32(127.0), np.float32(1e-8)).astype(np.float32)

    def rounded(q):
        return np.trunc(np.where(q >= 0, q + np.float32(0.5), q - np.float32(0.5)).astype(np.float32))

    want = rounded((xf / s[:, None]).astype(np.float32)).astype(np.int8)
    assert np.array_equal(codes, want)
    assert np.array_equal(scales, s.astype(np.float16).view(np.uint16))
    assert set(np.unique(np.abs(want[:, 1:]))) == {63, 64}  # both sides of the boundary occur
    by_product = rounded((xf * (np.float32(1.0) / s)[:, None]).astype(np.float32)).astype(np.int8)
    assert not np.array_equal(by_product, want)


def test_int8_store_scale_layout_head_major():
    """A token's scale for head g sits at [block][g][offset]; its codes at [block][offset][g]."""
    nb, bs, hkv, d = 3, 4, 2, 8
    kc = np.zeros((nb, bs, hkv, d), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, hkv, bs), np.uint16)
    vs = np.zeros_like(ks)
    k = torch.zeros(1, hkv, d)
    k[0, 0, 0], k[0, 1, 0] = 127.0, 254.0  # scales 1.0 and 2.0
    k = k.to(torch.bfloat16)
    oracle.store_kvcache_int8(kc, vc, ks, vs, k, k, [2 * bs + 3])  # block 2, offset 3
    assert ks[2, 0, 3] == 0x3C00 and ks[2, 1, 3] == 0x4000
    assert kc[2, 3, 0, 0] == 127 and kc[2, 3, 1, 0] == 127
    assert np.count_nonzero(ks) == 2 and np.count_nonzero(kc) == 2


def test_int8_attention_matches_brute_force_on_dequantised_cache():
    c = _identity_case(43, num_seqs=3, hq=4, hkv=2, d=16, bs=4, max_len=20, cached=True)
    nb, bs, hkv, d = c["pool_k"].shape
    kc8, ks = oracle.quantize_rows(c["pool_k"])  # scales [nb, bs, hkv]
    vc8, vs = oracle.quantize_rows(c["pool_v"])
    # cache scales are head-major inside a block: [nb, hkv, bs]
    kc8, vc8 = kc8.copy(), vc8.copy()
    ks, vs = np.ascontiguousarray(ks.transpose(0, 2, 1)), np.ascontiguousarray(vs.transpose(0, 2, 1))
    slots = oracle.slot_mapping(c["lens"], c["qlens"], c["blocks"], bs)
    oracle.store_kvcache_int8(kc8, vc8, ks, vs, c["k"], c["v"], slots)
    out, _ = oracle.paged_attention_int8(c["q"], kc8, vc8, ks, vs, c["lens"], c["qlens"], c["blocks"], bs, c["scale"])
    # independent dequantisation: numpy's fp16 -> fp32, identity block layout (plain slices)
    ksd = ks.transpose(0, 2, 1).view(np.float16).astype(np.float64)
    vsd = vs.transpose(0, 2, 1).view(np.float16).astype(np.float64)
    kd = (kc8.astype(np.float64) * ksd[..., None]).reshape(-1, hkv, d)
    vd = (vc8.astype(np.float64) * vsd[..., None]).reshape(-1, hkv, d)
    t0 = 0
    for b in range(3):
        lk, lq = int(c["lens"][b]), int(c["qlens"][b])
        s0 = int(c["starts"][b]) * bs
        qb = _f64(c["q"][t0:t0 + lq]).tolist()
        ref = np.array(brute.attention(qb, kd[s0:s0 + lk].tolist(), vd[s0:s0 + lk].tolist(), c["scale"]))
        np.testing.assert_allclose(out[t0:t0 + lq], ref, rtol=0, atol=1e-12)
        t0 += lq


def _nearest_bf16(p: float) -> float:
    """The bf16 value nearest to p (exact in fp32), ties to the even significand, found by
    comparing the distances to the two bf16 neighbours that bracket it."""
    if p == 0.0:
        return 0.0
    bits = int(np.array([abs(p)], np.float32).view(np.uint32)[0])
    lo = bits & 0xFFFF0000
    cands = [lo, lo + 0x10000]
    vals = [float(np.array([c], np.uint32).view(np.float32)[0]) for c in cands]
    dist = [abs(v - abs(p)) for v in vals]
    if dist[0] < dist[1] or (dist[0] == dist[1] and (cands[0] >> 16) % 2 == 0):
        r = vals[0]
    else:
        r = vals[1]
    return math.copysign(r, p)


def test_int8_bf16_values_are_the_nearest_bf16_of_code_times_scale():
    """The prefill reading of an INT8 cache ("面试问答准备: nano-vLLM 推理引擎优化", Q3: values x token
    scales in fp32, cast to the model's dtype): every code -127..127 against fp16 scales that are
    normal, subnormal, 1 and 3 (code x 3 has up to nine significant bits, so exact ties occur),
    each equal to the bf16 neighbour nearest the exact product; the exact reading is the product."""
    scales16 = np.array([1.0, 3.0, 1 / 127, 0.0123, 2.0 ** -20, 5.96e-8, 0.5 + 2.0 ** -10, 1000.0], np.float16)
    codes = np.arange(-127, 128, dtype=np.int8)
    nb, bs, hkv, d = len(scales16), 1, 1, codes.size
    kc = np.broadcast_to(codes, (nb, bs, hkv, d)).copy()
    ks = scales16.view(np.uint16).reshape(nb, hkv, bs).copy()
    got_bf16 = oracle.gather_dense_int8(kc, ks, nb, np.arange(nb), bs, values="bf16")
    got_exact = oracle.gather_dense_int8(kc, ks, nb, np.arange(nb), bs, values="exact")
    ties = 0
    for j in range(nb):
        s = float(scales16[j])
        for i, c in enumerate(codes.tolist()):
            p = c * s  # exact: 8 x 11 significant bits
            assert got_exact[j, 0, i] == p
            want = _nearest_bf16(p)
            assert got_bf16[j, 0, i] == want, (c, s, got_bf16[j, 0, i], want)
            f = np.array([abs(p)], np.float32).view(np.uint32)[0]
            ties += int(p != 0 and (f & 0xFFFF) == 0x8000)
    assert ties > 0


def test_int8_prefill_reading_is_attention_over_bf16_rounded_values():
    """paged_attention_int8(values="bf16") is the bf16-cache attention over code x scale rounded to
    bf16 (torch's fp32 -> bf16 conversion), and values="exact" differs from it."""
    c = _identity_case(47, num_seqs=3, hq=4, hkv=2, d=16, bs=4, max_len=20, cached=True)
    nb, bs, hkv, d = c["pool_k"].shape
    kc8, ks = oracle.quantize_rows(c["pool_k"] * 7)
    vc8, vs = oracle.quantize_rows(c["pool_v"] * 7)
    kc8, vc8 = kc8.copy(), vc8.copy()
    ks, vs = np.ascontiguousarray(ks.transpose(0, 2, 1)), np.ascontiguousarray(vs.transpose(0, 2, 1))
    args = (c["q"], kc8, vc8, ks, vs, c["lens"], c["qlens"], c["blocks"], bs, c["scale"])
    got, _ = oracle.paged_attention_int8(*args, values="bf16")
    exact, _ = oracle.paged_attention_int8(*args)

    def rounded(codes, sc):
        s = torch.from_numpy(sc.transpose(0, 2, 1).copy().view(np.float16)).float()
        return (torch.from_numpy(codes).float() * s[..., None]).to(torch.bfloat16)

    want, _ = oracle.paged_attention(c["q"], rounded(kc8, ks), rounded(vc8, vs), c["lens"], c["qlens"], c["blocks"],
                                     bs, c["scale"])
    np.testing.assert_array_equal(got, want)
    assert not np.array_equal(got, exact)
