"""pa_prefill_varlen_fused (store of the new tokens + prefill in one launch) on the GPU.

Checked three ways: the whole cache after the call equals the oracle's store
bit for bit; the output is within the oracle tolerance (max |err| <= 2e-2,
relative RMS <= 1e-2); and it is bitwise the output of pa_store_kvcache +
pa_prefill_varlen (the fused launch reads the new keys from the inputs, the
same bf16 values the store writes, and computes the same arithmetic).

Method: "手搓 vLLM 推理引擎", Step 4 (store_kvcache before the attention call).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, bits, dims_of, run_gpu_batch

pytestmark = pytest.mark.gpu


def _fused(w, batch, kc, vc):
    dims = dims_of(w, batch)
    dev = kc.device
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload(dev)
    out = torch.full_like(q, float("nan"))
    pa.pa_prefill_varlen_fused(dims, q, k, v, kc, vc, plan, batch.scale, out)
    return out, plan


def _run(w, row_select=None, compare_separate=True):
    """Every batch in order: prefill batches through the fused call (decode batches as usual);
    the oracle alongside; the separate two-launch path on its own cache copy."""
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    kc2, vc2 = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    ok_, ov_ = bits(w.pool.k_cache), bits(w.pool.v_cache)
    res = []
    for batch in w.batches:
        if batch.kind == "prefill":
            out, plan = _fused(w, batch, kc, vc)
        else:
            out, plan = run_gpu_batch(w, batch, kc, vc)
        sep = run_gpu_batch(w, batch, kc2, vc2)[0] if compare_separate else None
        sel = row_select(batch) if callable(row_select) else row_select
        ref, _ = oracle.run_batch(ok_, ov_, batch, w.pool.block_size, row_select=sel)
        res.append((batch, out, sep, ref, plan, sel))
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert np.array_equal(bits(kc), ok_), f"{w.name}: K cache differs from the oracle's store"
    assert np.array_equal(bits(vc), ov_), f"{w.name}: V cache differs from the oracle's store"
    return res


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefill_32", "qwen3_prefill_128", "qwen3_prefill_256",
                                  "qwen3_prefix", "qwen3_chunked"])
def test_fused_prefill_configs(name):
    """Configs with and without cached prefixes (qwen3_chunked: prefixes ending inside a block)."""
    w = workloads.make(name, device="cuda")
    for batch, out, sep, ref, plan, _ in _run(w):
        if batch.kind == "prefill":
            assert_close(out, ref, what=f"fused {name} (prefix_aligned={plan.meta.prefix_aligned})")
            assert torch.equal(out, sep), f"{name}: fused output differs from store + prefill"


FUSED_CASES = [  # seed, num_seqs, hq, hkv, d, bs, max_len, cached
    (701, 3, 2, 1, 64, 16, 300, None),
    (702, 4, 8, 2, 128, 16, 700, "aligned"),
    (703, 5, 14, 2, 128, 32, 900, "aligned"),
    (704, 4, 4, 4, 64, 256, 700, "aligned"),
    (705, 6, 28, 4, 128, 16, 520, "random"),
    (706, 2, 16, 8, 128, 128, 1300, "aligned"),
    # cached prefixes ending anywhere (the straddling key box patched from the inputs)
    (707, 5, 28, 4, 128, 16, 700, "random"),
    (708, 4, 16, 8, 128, 256, 1500, "random"),
    (709, 3, 8, 2, 64, 1024, 2100, "random"),
    (710, 6, 14, 2, 128, 64, 900, "random"),
    (711, 7, 7, 1, 64, 32, 400, "random"),
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=[str(c[0]) for c in FUSED_CASES])
def test_fused_prefill_random(case):
    seed, ns, hq, hkv, d, bs, ml, cached = case
    w = workloads.random_case(seed, num_seqs=ns, hq=hq, hkv=hkv, d=d, bs=bs, max_len=ml, cached=cached,
                              device="cuda")
    (batch, out, sep, ref, plan, _), = _run(w)
    if cached != "random":
        assert plan.meta.prefix_aligned == 1
    assert_close(out, ref, what=f"fused case {seed}")
    assert torch.equal(out, sep), f"case {seed}: fused output differs from store + prefill"


def test_fused_prefill_qwen25_every_row():
    """The benched 4 x 4096 prompt batch: one launch (no prefix), every row against the oracle."""
    w = workloads.make("qwen25_prefill", device="cuda")
    (batch, out, sep, ref, plan, _), = _run(w)
    assert plan.meta.prefix_aligned == 1
    assert_close(out, ref, what="fused qwen25 prefill (every row)")
    assert torch.equal(out, sep)


def test_fused_prefill_decode_rows():
    """Lq = 1 rows (decode steps run through the prefill) whose cached prefixes are whole blocks."""
    hq, hkv, d, bs = 8, 2, 128, 16
    lens = np.array([33, 129, 17, 257], np.int32)  # prefixes 32, 128, 16, 256
    nb = int(sum(-(-int(l) // bs) for l in lens)) + 2
    perm = np.random.default_rng(41).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(42)
    mk = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = len(lens)
    batch = workloads.Batch("prefill", lens, np.ones(t, np.int32), blocks, mk(t, hq, d), mk(t, hkv, d),
                            mk(t, hkv, d), hq, d ** -0.5)
    (batch, out, sep, ref, plan, _), = _run(workloads.Workload("fused_decode_rows", pool, [batch]))
    assert plan.meta.prefix_aligned == 1
    assert_close(out, ref, what="fused decode rows")
    assert torch.equal(out, sep)


def test_fused_prefill_edge_lengths():
    """Sequences without new tokens, single tokens, exact tiles and block-aligned prefixes in one batch."""
    hq, hkv, d, bs = 4, 2, 128, 16
    lens = np.array([16, 17, 48, 129, 5, 128, 256], np.int32)
    qlens = np.array([0, 1, 16, 129, 0, 128, 96], np.int32)  # prefixes 16, 16, 32, 0, -, 0, 160
    nb = int(sum(-(-int(l) // bs) for l in lens)) + 2
    perm = np.random.default_rng(19).permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for l in lens:
        n = -(-int(l) // bs)
        blocks.append(perm[o:o + n])
        o += n
    g = torch.Generator(device="cuda").manual_seed(20)
    mk = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)
    pool = workloads.Pool(nb, bs, hkv, d, mk(nb, bs, hkv, d), mk(nb, bs, hkv, d))
    t = int(qlens.sum())
    batch = workloads.Batch("prefill", lens, qlens, blocks, mk(t, hq, d), mk(t, hkv, d), mk(t, hkv, d), hq, d ** -0.5)
    (batch, out, sep, ref, plan, _), = _run(workloads.Workload("fused_edges", pool, [batch]))
    assert plan.meta.prefix_aligned == 1
    assert_close(out, ref, what="fused edges")
    assert torch.equal(out, sep)


def test_fused_prefill_bad_slot_flagged():
    """A slot outside [-1, num_slots) is skipped and flagged (bit 0); -1 skips silently; the other
    rows are stored and the attention reads the new keys from the inputs either way."""
    w = workloads.random_case(711, num_seqs=2, hq=4, hkv=2, d=128, bs=16, max_len=200, cached=None, device="cuda")
    batch = w.batches[0]
    dims = dims_of(w, batch)
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
    slots = plan.dev[plan.meta.off_slot_mapping:plan.meta.off_slot_mapping + 4 * batch.num_tokens].view(torch.int32)
    orig = slots.clone()
    num_slots = w.pool.num_blocks * w.pool.block_size
    slots[3] = num_slots + 5
    slots[7] = -1
    q, k, v = batch.q.cuda(), batch.k.cuda(), batch.v.cuda()
    out = torch.empty_like(q)
    pa.pa_prefill_varlen_fused(dims, q, k, v, kc, vc, plan, batch.scale, out)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() & 1
    n, hkv, d = num_slots, w.pool.num_kv_heads, w.pool.head_dim
    flat = kc.view(n, hkv, d)
    before = w.pool.k_cache.view(n, hkv, d)
    for t in range(batch.num_tokens):
        s = int(orig[t])
        if t in (3, 7):
            assert torch.equal(flat[s], before[s]), f"row {t} was written"
        else:
            assert torch.equal(flat[s], k[t]), f"row {t} not stored"
    # the attention does not depend on the cache rows of new keys: same output as the clean call
    kc2, vc2 = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    slots.copy_(orig)
    out2 = torch.empty_like(q)
    pa.pa_prefill_varlen_fused(dims, q, k, v, kc2, vc2, plan, batch.scale, out2)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert torch.equal(out, out2)


def test_fused_prefill_replayed_from_a_cuda_graph():
    """Captured once, replayed on new inputs copied into the captured buffers: the same output and
    cache as eager calls (no host synchronisation or allocation inside the call)."""
    w = workloads.random_case(721, num_seqs=3, hq=8, hkv=2, d=128, bs=16, max_len=600, cached="aligned",
                              device="cuda")
    batch = w.batches[0]
    dims = dims_of(w, batch)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
    assert plan.meta.prefix_aligned == 1
    q, k, v = batch.q.clone(), batch.k.clone(), batch.v.clone()
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.pa_prefill_varlen_fused(dims, q, k, v, kc, vc, plan, batch.scale, out, stream=s)  # set-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.pa_prefill_varlen_fused(dims, q, k, v, kc, vc, plan, batch.scale, out,
                                   stream=torch.cuda.current_stream())
    g = torch.Generator(device="cuda").manual_seed(722)
    for _ in range(2):
        nq = torch.randn(q.shape, device="cuda", generator=g).to(torch.bfloat16)
        nk = torch.randn(k.shape, device="cuda", generator=g).to(torch.bfloat16)
        nv = torch.randn(v.shape, device="cuda", generator=g).to(torch.bfloat16)
        q.copy_(nq), k.copy_(nk), v.copy_(nv)
        graph.replay()
        kc2, vc2 = w.pool.k_cache.clone(), w.pool.v_cache.clone()
        ref = torch.empty_like(q)
        pa.pa_prefill_varlen_fused(dims, nq, nk, nv, kc2, vc2, plan, batch.scale, ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        sm = plan.host_array(plan.meta.off_slot_mapping, batch.num_tokens)
        n = w.pool.num_blocks * w.pool.block_size
        assert torch.equal(kc.view(n, -1)[torch.as_tensor(sm, device="cuda").long()], nk.view(batch.num_tokens, -1))
        assert torch.equal(kc.view(n, -1)[torch.as_tensor(sm, device="cuda").long()],
                           kc2.view(n, -1)[torch.as_tensor(sm, device="cuda").long()])
    assert pa.pa_read_device_error() == 0


def _launches(fn, stream):
    """Nodes of the graph that stream capture of fn() records (each launch is one node)."""
    import ctypes
    import glob
    import os
    rt = None
    cands = ["libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"]
    cands += glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart*.so*"))
    for c in cands:
        try:
            rt = ctypes.CDLL(c)
            break
        except OSError:
            continue
    if rt is None:
        pytest.skip("no CUDA runtime library to capture with")
    h = ctypes.c_void_p(stream.cuda_stream)
    assert rt.cudaStreamBeginCapture(h, 2) == 0  # relaxed capture mode
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        rc = rt.cudaStreamEndCapture(h, ctypes.byref(graph))
    assert rc == 0
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    rt.cudaGraphDestroy(graph)
    return n.value


def test_fused_prefill_unaligned_prefixes_are_one_launch():
    """The chunked-prefill batch (prefixes ~ U{0..1024}, block 256): the call records one launch
    (stream capture), the cache equals the oracle's store and the output is bitwise the
    two-launch one."""
    w = workloads.make("qwen3_chunked", device="cuda")
    batch = w.batches[0]
    dims = dims_of(w, batch)
    plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists).upload("cuda")
    assert plan.meta.prefix_aligned == 0
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    out = torch.empty_like(batch.q)
    pa.pa_prefill_varlen_fused(dims, batch.q, batch.k, batch.v, kc, vc, plan, batch.scale, out)  # warm-up
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    n = _launches(lambda: pa.pa_prefill_varlen_fused(dims, batch.q, batch.k, batch.v, kc, vc, plan, batch.scale, out,
                                                     stream=s), s)
    assert n == 1, f"{n} launches"
    (b, out2, sep, ref, _, _), = _run(w)
    assert torch.equal(out, out2) and torch.equal(out, sep)
    assert_close(out, ref, what="fused qwen3 chunked (one launch)")
