"""Seeded synthetic inputs for paged KV-cache attention.

This module holds data only: random values, sequence lengths and physical-block
assignments.  It computes nothing of the attention method (no slot arithmetic,
no prefix sums, no softmax); both the CUDA library's tests/bench and the CPU
oracle receive exactly the arrays built here and derive everything else on
their own.

Shapes follow the pages' workloads:

* ``tiny``            2 sequences (37, 64 tokens), 2 q heads / 1 KV head, D 64,
                      block 16, 16-block pool, seed 0 (prefill, then one decode
                      step per sequence).
* ``qwen3_prefill_N`` Qwen3-0.6B attention (16 q / 8 KV heads, D 128, block 256),
                      8 sequences of N in {32, 128, 256} tokens over a permuted
                      64-block pool.
* ``qwen3_decode``    256 sequences, one new token each, context = in + out with
                      in, out ~ U{100..1024}, pool sized to fit, permuted.
* ``qwen3_prefix``    8 x (44 new of 300), block 0 physically shared by all 8.
* ``qwen3_chunked``   16 sequences, cached prefix ~ U{0..1024}, new chunk ~ U{1..512}.
* ``qwen25_prefill``  Qwen2.5-7B attention (28 q / 4 KV heads, D 128, block 16),
                      4 x 4096 causal prefill.
* ``qwen25_decode``   64 sequences at context 32768 over a fully permuted
                      131072-block pool.

Values are N(0, 1) drawn in fp32 and rounded to bf16.  Metadata (lengths,
permutations) always comes from a CPU generator so it is identical on every
machine; values come from a generator on the requested device.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch


@dataclass
class Pool:
    """Physical KV-cache pool, layout [num_blocks, block_size, num_kv_heads, head_dim]."""
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    k_cache: torch.Tensor   # bf16, initial contents (cached prefixes + canary)
    v_cache: torch.Tensor


@dataclass
class Batch:
    """One attention call: per-sequence lengths, block lists and new-token tensors.

    ``seq_lens[b]`` is the total key length after this call's tokens are stored,
    ``query_lens[b]`` the number of new (queried) tokens at its end.  The first
    ``seq_lens - query_lens`` tokens are already in the pool.
    """
    kind: str                      # "prefill" or "decode"
    seq_lens: np.ndarray           # int32 [B]
    query_lens: np.ndarray         # int32 [B]
    block_lists: List[np.ndarray]  # int32 physical block ids per sequence
    q: torch.Tensor                # bf16 [sum(query_lens), Hq, D]
    k: torch.Tensor                # bf16 [sum(query_lens), Hkv, D]
    v: torch.Tensor                # bf16 [sum(query_lens), Hkv, D]
    num_heads: int
    scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())


@dataclass
class Workload:
    name: str
    pool: Pool
    batches: List[Batch] = field(default_factory=list)


def _values(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _pool_values(gen: torch.Generator, nb: int, bs: int, hkv: int, d: int, device) -> torch.Tensor:
    """N(0,1) bf16 pool drawn in chunks so the fp32 temporary stays small."""
    out = torch.empty((nb, bs, hkv, d), dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _gens(seed: int, device):
    meta = torch.Generator(device="cpu").manual_seed(seed)
    dev = torch.device(device)
    vals = torch.Generator(device=dev).manual_seed(seed + 7919)
    return meta, vals, dev


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _batch(kind, seq_lens, query_lens, block_lists, hq, hkv, d, vals, dev) -> Batch:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int32)
    t = int(query_lens.sum())
    q = _values(vals, (t, hq, d), dev)
    k = _values(vals, (t, hkv, d), dev)
    v = _values(vals, (t, hkv, d), dev)
    return Batch(kind, seq_lens, query_lens, [np.asarray(b, dtype=np.int32) for b in block_lists],
                 q, k, v, hq, 1.0 / float(np.sqrt(d)))


def tiny(device="cpu") -> Workload:
    """2 sequences (37, 64), Hq 2 / Hkv 1, D 64, block 16, pool 16, seed 0."""
    meta, vals, dev = _gens(0, device)
    nb, bs, hq, hkv, d = 16, 16, 2, 1, 64
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    lens = [37, 64]
    pre_blocks = [perm[0:3], perm[3:7]]
    prefill = _batch("prefill", lens, lens, pre_blocks, hq, hkv, d, vals, dev)
    # decode: one more token each; seq 1 (65 tokens) needs a fifth block
    dec_blocks = [perm[0:3], np.concatenate([perm[3:7], perm[7:8]])]
    decode = _batch("decode", [38, 65], [1, 1], dec_blocks, hq, hkv, d, vals, dev)
    return Workload("tiny", pool, [prefill, decode])


def qwen3_prefill(n: int, device="cpu") -> Workload:
    """Qwen3-0.6B attention, 8 sequences x n new tokens, permuted 64-block pool."""
    meta, vals, dev = _gens(2, device)
    nb, bs, hq, hkv, d = 64, 256, 16, 8, 128
    assert n <= bs
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    blocks = [perm[i:i + 1] for i in range(8)]
    return Workload(f"qwen3_prefill_{n}", pool, [_batch("prefill", [n] * 8, [n] * 8, blocks, hq, hkv, d, vals, dev)])


def qwen3_decode(device="cpu", num_seqs: int = 256) -> Workload:
    """256 decode sequences, context = in + out, in/out ~ U{100..1024}, block 256."""
    meta, vals, dev = _gens(3, device)
    bs, hq, hkv, d = 256, 16, 8, 128
    inp = torch.randint(100, 1025, (num_seqs,), generator=meta)
    outp = torch.randint(100, 1025, (num_seqs,), generator=meta)
    ctx = (inp + outp).numpy().astype(np.int32)
    need = [_ceil_div(int(c), bs) for c in ctx]
    nb = int(sum(need))
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    blocks, o = [], 0
    for n in need:
        blocks.append(perm[o:o + n])
        o += n
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    return Workload("qwen3_decode", pool, [_batch("decode", ctx, np.ones(num_seqs, np.int32), blocks, hq, hkv, d, vals, dev)])


def qwen3_prefix(device="cpu") -> Workload:
    """8 x 300-token sequences, first block (256 tokens) physically shared, last 44 queried."""
    meta, vals, dev = _gens(4, device)
    nb, bs, hq, hkv, d = 64, 256, 16, 8, 128
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    shared = perm[0]
    blocks = [np.array([shared, perm[1 + b]], np.int32) for b in range(8)]
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    return Workload("qwen3_prefix", pool, [_batch("prefill", [300] * 8, [44] * 8, blocks, hq, hkv, d, vals, dev)])


def qwen3_chunked(device="cpu", num_seqs: int = 16) -> Workload:
    """16 sequences, cached prefix ~ U{0..1024}, new chunk ~ U{1..512}, private blocks."""
    meta, vals, dev = _gens(44, device)
    bs, hq, hkv, d = 256, 16, 8, 128
    prefix = torch.randint(0, 1025, (num_seqs,), generator=meta).numpy().astype(np.int32)
    chunk = torch.randint(1, 513, (num_seqs,), generator=meta).numpy().astype(np.int32)
    lens = prefix + chunk
    need = [_ceil_div(int(c), bs) for c in lens]
    nb = int(sum(need))
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    blocks, o = [], 0
    for n in need:
        blocks.append(perm[o:o + n])
        o += n
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    return Workload("qwen3_chunked", pool, [_batch("prefill", lens, chunk, blocks, hq, hkv, d, vals, dev)])


def qwen25_prefill(device="cpu", num_seqs: int = 4, seq_len: int = 4096) -> Workload:
    """Qwen2.5-7B attention (28 q / 4 KV heads, D 128, block 16), 4 x 4096 causal prefill."""
    meta, vals, dev = _gens(5, device)
    bs, hq, hkv, d = 16, 28, 4, 128
    per = _ceil_div(seq_len, bs)
    nb = per * num_seqs
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    blocks = [perm[b * per:(b + 1) * per] for b in range(num_seqs)]
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    lens = [seq_len] * num_seqs
    return Workload("qwen25_prefill", pool, [_batch("prefill", lens, lens, blocks, hq, hkv, d, vals, dev)])


def qwen25_decode(device="cpu", num_seqs: int = 64, ctx: int = 32768) -> Workload:
    """64 decode sequences at context 32768 over a fully permuted pool (block 16)."""
    meta, vals, dev = _gens(55, device)
    bs, hq, hkv, d = 16, 28, 4, 128
    per = _ceil_div(ctx, bs)
    nb = per * num_seqs
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    blocks = [perm[b * per:(b + 1) * per] for b in range(num_seqs)]
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    return Workload("qwen25_decode", pool,
                    [_batch("decode", [ctx] * num_seqs, [1] * num_seqs, blocks, hq, hkv, d, vals, dev)])


def random_case(seed: int, *, num_seqs: int, hq: int, hkv: int, d: int, bs: int,
                max_len: int, kind: str = "prefill", extra_blocks: int = 3,
                device="cpu", min_len: int = 1, cached: Optional[str] = "random") -> Workload:
    """Small random varlen case for parity sweeps.

    Lengths ~ U{min_len..max_len}; for prefill, the cached prefix is either 0
    (``cached=None``), ~ U{0..len-1} (``"random"``) or that rounded down to a
    multiple of min(bs, 128) (``"aligned"``, whole cached blocks); for decode,
    every sequence queries its last token.  Blocks are a random permutation of a pool with a few spare
    blocks that stay untouched (canary).
    """
    meta, vals, dev = _gens(seed, device)
    lens = torch.randint(min_len, max_len + 1, (num_seqs,), generator=meta).numpy().astype(np.int32)
    if kind == "decode":
        qlens = np.ones(num_seqs, np.int32)
    elif cached is None:
        qlens = lens.copy()
    else:
        pre = np.array([int(torch.randint(0, int(l), (1,), generator=meta)) for l in lens], np.int32)
        if cached == "aligned":
            pre -= pre % min(bs, 128)
        qlens = (lens - pre).astype(np.int32)
    need = [_ceil_div(int(c), bs) for c in lens]
    nb = int(sum(need)) + extra_blocks
    perm = torch.randperm(nb, generator=meta).numpy().astype(np.int32)
    blocks, o = [], 0
    for n in need:
        blocks.append(perm[o:o + n])
        o += n
    pool = Pool(nb, bs, hkv, d, _pool_values(vals, nb, bs, hkv, d, dev), _pool_values(vals, nb, bs, hkv, d, dev))
    return Workload(f"random_{seed}", pool, [_batch(kind, lens, qlens, blocks, hq, hkv, d, vals, dev)])


WORKLOADS = {
    "tiny": tiny,
    "qwen3_prefill_32": lambda device="cpu": qwen3_prefill(32, device),
    "qwen3_prefill_128": lambda device="cpu": qwen3_prefill(128, device),
    "qwen3_prefill_256": lambda device="cpu": qwen3_prefill(256, device),
    "qwen3_decode": qwen3_decode,
    "qwen3_prefix": qwen3_prefix,
    "qwen3_chunked": qwen3_chunked,
    "qwen25_prefill": qwen25_prefill,
    "qwen25_decode": qwen25_decode,
}


def make(name: str, device="cpu") -> Workload:
    return WORKLOADS[name](device=device)
