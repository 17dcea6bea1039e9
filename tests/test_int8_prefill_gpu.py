"""INT8 prefill on the GPU against the oracle's attention over the dequantised cache.

Method: "面试问答准备: nano-vLLM 推理引擎优化", Q3 — per-(token, KV head) INT8
codes with fp16 scales; the prefill reads the keys and values its batch
references as code x token scale rounded to bf16 (a gather launch into a
scratch cache) and runs the bf16 attention over them.  Tolerances as for the
bf16 path: max |err| <= 2e-2, relative RMS <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, dims_of, int8_equal, int8_pools, run_gpu_batch_int8, sample_rows

pytestmark = pytest.mark.gpu


def _run_both(w, row_select=None):
    """Every batch in order on both sides (store, then attention); the caches must stay bit-identical."""
    gpu, host = int8_pools(w, w.batches[0].num_heads)
    res = []
    for batch in w.batches:
        out, _ = run_gpu_batch_int8(w, batch, gpu)
        sel = row_select(batch) if callable(row_select) else row_select
        ref, _ = oracle.run_batch_int8(*host, batch, w.pool.block_size, row_select=sel)
        res.append((batch, out, ref, sel))
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(gpu, host, what=w.name)
    return res


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefill_32", "qwen3_prefill_128", "qwen3_prefill_256",
                                  "qwen3_prefix", "qwen3_chunked"])
def test_int8_prefill_configs(name):
    """Prefill (and, for the tiny case, the decode step after it) on the INT8 cache."""
    for batch, out, ref, _ in _run_both(workloads.make(name, device="cuda")):
        assert_close(out, ref, what=f"int8 {name} {batch.kind}")


CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (501, 3, 2, 1, 64, 16, 300, None),
    (502, 4, 4, 2, 64, 256, 700, "random"),
    (503, 5, 7, 1, 128, 16, 400, "random"),
    (504, 3, 14, 2, 128, 256, 520, None),
    (505, 6, 8, 8, 128, 16, 260, "random"),
    (506, 2, 16, 1, 64, 32, 390, "random"),
    (507, 4, 28, 4, 128, 16, 333, "random"),
    (508, 3, 16, 8, 128, 1024, 1100, "random"),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_int8_prefill_random(case):
    seed, B, hq, hkv, d, bs, max_len, cached = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, device="cuda",
                              cached=cached)
    (batch, out, ref, _), = _run_both(w)
    assert_close(out, ref, what=f"int8 case {seed}")


# Many more work items than SMs: every CTA of the persistent kernel runs several
# items back to back (code and factor rings, query refills and conversions
# carried across items).
MULTI = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (521, 160, 4, 4, 128, 16, 512, "random"),
    (522, 96, 16, 4, 64, 32, 300, "random"),
    (523, 48, 28, 4, 128, 16, 200, None),
    (524, 200, 16, 8, 128, 256, 300, "random"),
]


@pytest.mark.parametrize("case", MULTI, ids=[str(c[0]) for c in MULTI])
def test_int8_prefill_many_items_per_cta(case):
    seed, B, hq, hkv, d, bs, max_len, cached = case
    w = workloads.random_case(seed, num_seqs=B, hq=hq, hkv=hkv, d=d, bs=bs, max_len=max_len, device="cuda",
                              cached=cached)
    b = w.batches[0]
    items = pa.pa_pack_prefill(dims_of(w, b), b.seq_lens, b.query_lens, b.block_lists, pin=False).meta.num_tiles
    assert items > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    (batch, out, ref, _), = _run_both(w)
    assert_close(out, ref, what=f"int8 case {seed}, {items} items")


def test_int8_prefill_edge_lengths():
    """Sequences with no new tokens, single-token sequences and exact-tile lengths in one batch."""
    hq, hkv, d, bs = 4, 2, 128, 16
    lens = np.array([1, 17, 40, 129, 5, 128, 256], np.int32)
    qlens = np.array([1, 0, 1, 129, 0, 128, 100], np.int32)
    nb = int(sum(-(-l // bs) for l in lens)) + 2
    perm = np.random.default_rng(9).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(10)
    mk = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = int(qlens.sum())
    batch = workloads.Batch("prefill", lens, qlens, blocks, mk(t, hq, d), mk(t, hkv, d), mk(t, hkv, d), hq, d ** -0.5)
    (batch, out, ref, _), = _run_both(workloads.Workload("int8_edges", pool, [batch]))
    assert_close(out, ref, what="int8 edges")


def test_int8_prefill_qwen25_every_row():
    """Qwen2.5-7B attention shape, 4 x 4096 causal prefill (the measured workload), every row."""
    w = workloads.make("qwen25_prefill", device="cuda")
    (batch, out, ref, _), = _run_both(w)
    assert_close(out, ref, what="int8 qwen25 prefill (every row)")


def test_int8_prefill_single_32k_sequence_sampled():
    """One 32768-token causal prompt on the INT8 cache: items of up to 256 key tiles (code,
    factor and release rings wrapping many times); sampled rows."""
    w = workloads.random_case(561, num_seqs=1, hq=28, hkv=4, d=128, bs=16, min_len=32768, max_len=32768,
                              cached=None, device="cuda")
    (batch, out, ref, sel), = _run_both(w, row_select=lambda b: sample_rows(b, 24, seed=9))
    assert_close(out, ref, rows=sel, what="int8 single 32k prefill (sampled rows)")


def test_int8_prefill_and_decode_over_mixed_token_magnitudes():
    """Tokens whose K/V magnitudes span 1e-4 .. 10^0.5 (scales down to ~1e-6, so that the
    decode's fp16 code x scale products fall in the subnormal range, and up to about 3x
    those of N(0, 1) data) and all-zero tokens (scale 0): a prefill over them, then a
    decode of each sequence's last token."""
    hq, hkv, d, bs = 8, 2, 128, 16
    lens = np.array([300, 77, 129], np.int32)
    nb = int(sum(-(-l // bs) for l in lens)) + 3
    perm = np.random.default_rng(31).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(32)

    def kv(*shape):  # rows scaled by 10^U(-4, 0.5) per (token, head); one row in 9 all zero
        x = torch.randn(*shape, device="cuda", generator=g)
        mag = 10.0 ** (torch.rand(*shape[:-1], 1, device="cuda", generator=g) * 4.5 - 4.0)
        zero = torch.rand(*shape[:-1], 1, device="cuda", generator=g) < 1 / 9
        return (x * mag).masked_fill(zero, 0.0).to(torch.bfloat16)

    pool = workloads.Pool(nb, bs, hkv, d, kv(nb, bs, hkv, d), kv(nb, bs, hkv, d))
    t = int(lens.sum())
    q = torch.randn(t, hq, d, device="cuda", generator=g).to(torch.bfloat16)
    pre = workloads.Batch("prefill", lens, lens.copy(), blocks, q, kv(t, hkv, d), kv(t, hkv, d), hq, d ** -0.5)
    last = np.cumsum(lens) - 1
    dec = workloads.Batch("decode", lens, np.ones(3, np.int32), blocks, pre.q[last], pre.k[last], pre.v[last], hq,
                          d ** -0.5)
    for batch, out, ref, _ in _run_both(workloads.Workload("int8_magnitudes", pool, [pre, dec])):
        assert_close(out, ref, what=f"int8 mixed magnitudes {batch.kind}")


def test_int8_prefill_matches_int8_decode():
    """Decode at context n equals row n-1 of an INT8 prefill over the same n tokens (same cache)."""
    n, hq, hkv, d, bs = 777, 14, 2, 128, 16
    w = workloads.random_case(13, num_seqs=1, hq=hq, hkv=hkv, d=d, bs=bs, min_len=n, max_len=n, device="cuda",
                              cached=None)
    batch = w.batches[0]
    gpu, _ = int8_pools(w, hq)
    out_p, _ = run_gpu_batch_int8(w, batch, gpu)
    dec = workloads.Batch("decode", batch.seq_lens, np.ones(1, np.int32), batch.block_lists, batch.q[-1:],
                          batch.k[-1:], batch.v[-1:], hq, batch.scale)
    out_d, _ = run_gpu_batch_int8(w, dec, gpu, split_tokens=128)
    torch.cuda.synchronize()
    a, b = out_p[-1].float(), out_d[0].float()
    assert (a - b).abs().max().item() < 1e-2


@pytest.mark.parametrize("seed,bs,hkv,d", [(881, 16, 2, 128), (882, 256, 8, 128), (883, 32, 4, 64)])
def test_int8_gather_scratch_is_code_times_scale_rounded_to_bf16(seed, bs, hkv, d):
    """The gather's output, read back from the workspace: for every key of every sequence with
    new tokens, the scratch row the plan's scratch tables give holds RN_bf16(code x fp16 scale)
    of the cache row its block table names, bit for bit against the oracle's prefill reading
    (a sequence without new tokens gets no scratch block)."""
    w = workloads.random_case(seed, num_seqs=7, hq=2 * hkv, hkv=hkv, d=d, bs=bs, max_len=700, cached="random",
                              device="cuda")
    b0 = w.batches[0]
    # sequence 2 without new tokens: its rows taken out of q/k/v
    qlens = b0.query_lens.copy()
    start = int(qlens[:2].sum())
    keep = torch.cat([torch.arange(start), torch.arange(start + int(qlens[2]), int(qlens.sum()))]).to(b0.q.device)
    qlens[2] = 0
    batch = workloads.Batch("prefill", b0.seq_lens, qlens, b0.block_lists, b0.q[keep], b0.k[keep], b0.v[keep],
                            b0.num_heads, b0.scale)
    gpu, host = int8_pools(w, batch.num_heads)
    out, plan = run_gpu_batch_int8(w, batch, gpu)
    slots = oracle.slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, bs)
    oracle.store_kvcache_int8(*host, batch.k, batch.v, slots)
    # the call above allocated its own workspace; run once more into a zeroed one this test keeps
    ws = torch.zeros(int(plan.meta.workspace_bytes), dtype=torch.uint8, device="cuda")
    pa.pa_prefill_varlen_int8(dims_of(w, batch), batch.q.cuda(), *gpu, plan, batch.scale, out, ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    int8_equal(gpu, host, what="gather case")
    m = plan.meta
    rows = m.scratch_blocks * 128
    scratch = ws.view(torch.bfloat16).view(2, rows, hkv, d).float().cpu().numpy().astype(np.float64)
    tab = plan.host_array(m.off_scratch_tables, len(batch.seq_lens) * m.scratch_pitch).reshape(-1, m.scratch_pitch)
    written = np.zeros(rows, bool)
    for b, (lk, lq) in enumerate(zip(batch.seq_lens, batch.query_lens)):
        lk, lq = int(lk), int(lq)
        if lq == 0:
            assert (tab[b] == -1).all()
            continue
        idx = np.concatenate([np.arange(128) + 128 * int(s) for s in tab[b][: -(-lk // 128)]])[:lk]
        written[idx] = True
        for t, (codes, scales) in enumerate(((host[0], host[2]), (host[1], host[3]))):
            want = oracle.gather_dense_int8(codes, scales, lk, batch.block_lists[b], bs, values="bf16")
            np.testing.assert_array_equal(scratch[t, idx], want, err_msg=f"sequence {b} tensor {t}")
    assert not scratch[:, ~written].any(), "rows past a sequence's end were written"
