"""CPU tests of the C ABI: the library loads, exports every declared entry point,
rejects bad arguments on the host, and packs metadata exactly as the oracle's
own definition does (integer work: bit-exact)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedattn.h")


def test_library_exports_every_declared_symbol():
    text = open(HEADER).read()
    declared = set(re.findall(r"^(?:int|const char \*)\s*(pa_\w+)\s*\(", text, flags=re.M))
    assert {"pa_store_kvcache", "pa_prefill_varlen", "pa_decode"} <= declared
    lib = pa.lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert set(pa.EXPORTS) == declared
    assert pa.pa_version() == 0x000500


def test_binding_argument_counts_match_the_header():
    """Every declaration's parameter count equals the binding's ctypes argument list, so a
    signature change in the header cannot leave the binding calling with the old layout."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    lib = pa.lib()
    checked = 0
    for name, params in re.findall(r"^(?:int|const char \*)\s*(pa_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes)
        checked += 1
    assert checked == len(pa.EXPORTS)


def test_struct_sizes_match_header_layout():
    assert ctypes.sizeof(pa.pa_dims) == 20
    assert ctypes.sizeof(pa.pa_prefill_meta) == 8 * 4 + 9 * 8 + 2 * 4
    # fields added after total_bytes leave the earlier offsets where they were
    assert pa.pa_prefill_meta.total_bytes.offset == 8 * 4 + 5 * 8
    assert ctypes.sizeof(pa.pa_decode_meta) == 6 * 4 + 7 * 8


@pytest.mark.parametrize("d,code", [((4, 16, 8, 3, 128), pa.PA_ERR_UNSUPPORTED),   # Hq % Hkv
                                    ((4, 16, 8, 2, 96), pa.PA_ERR_UNSUPPORTED),    # head_dim
                                    ((4, 24, 8, 2, 128), pa.PA_ERR_UNSUPPORTED),   # block_size not 2^k
                                    ((4, 8, 8, 2, 128), pa.PA_ERR_UNSUPPORTED),    # block_size < 16
                                    ((4, 16, 34, 2, 128), pa.PA_ERR_UNSUPPORTED),  # group 17 > 16
                                    ((4, 16, 0, 1, 128), pa.PA_ERR_INVALID_ARG)])
def test_dims_validation(d, code):
    dims = pa.make_dims(*d)
    meta = pa.pa_prefill_meta()
    rc = pa.lib().pa_pack_prefill(ctypes.byref(dims), 0, None, None, None, None, None, 0, ctypes.byref(meta))
    assert rc == code
    rc = pa.lib().pa_store_kvcache(ctypes.byref(dims), None, None, None, None, None, 1, None)
    assert rc == code


def test_device_calls_reject_bad_args_without_touching_the_gpu():
    dims = pa.make_dims(4, 16, 4, 2, 64)
    L = pa.lib()
    assert L.pa_store_kvcache(ctypes.byref(dims), None, None, None, None, None, 3, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache(ctypes.byref(dims), None, None, None, None, None, -1, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache(ctypes.byref(dims), None, None, None, None, None, 0, None) == pa.PA_OK
    assert L.pa_store_kvcache(ctypes.byref(dims), 8, 16, 32, 48, 64, 1, None) == pa.PA_ERR_INVALID_ARG  # misaligned
    meta = pa.pa_prefill_meta()
    meta.num_tiles, meta.total_q, meta.num_seqs, meta.max_blocks_per_seq, meta.rows_per_tile = 1, 1, 1, 1, 64
    assert L.pa_prefill_varlen(ctypes.byref(dims), None, None, None, None, None, None, ctypes.c_float(0.1),
                               None, ctypes.byref(meta), None, None) == pa.PA_ERR_INVALID_ARG
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        assert L.pa_prefill_varlen(ctypes.byref(dims), 16, 16, 16, 16, 16, 16, ctypes.c_float(bad), 16,
                                   ctypes.byref(meta), 16, None) == pa.PA_ERR_INVALID_ARG
    meta.rows_per_tile = 7  # packed for other dims
    assert L.pa_prefill_varlen(ctypes.byref(dims), 16, 16, 16, 16, 16, 16, ctypes.c_float(0.1), 16,
                               ctypes.byref(meta), 16, None) == pa.PA_ERR_INVALID_ARG
    dm = pa.pa_decode_meta()
    dm.num_items, dm.num_seqs, dm.max_blocks_per_seq, dm.max_splits = 1, 1, 1, 1
    dm.workspace_bytes = 1024
    assert L.pa_decode(ctypes.byref(dims), 16, 16, 16, 16, 16, ctypes.c_float(0.1), 16, ctypes.byref(dm), 16, 16,
                       None, 0, None) == pa.PA_ERR_WORKSPACE
    assert "workspace" in pa.pa_last_error_string()
    for bad in (0, 10000001):
        assert L.pa_selftest_bounded_wait(bad, 0, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_stream_read(16, 64, None, None) == pa.PA_ERR_INVALID_ARG     # no sink
    assert L.pa_stream_read(8, 64, 16, None) == pa.PA_ERR_INVALID_ARG       # src misaligned
    assert L.pa_stream_read(16, 40, 16, None) == pa.PA_ERR_INVALID_ARG      # bytes not a multiple of 16
    assert L.pa_stream_read(None, 16, 16, None) == pa.PA_ERR_INVALID_ARG    # no src
    assert L.pa_stream_read(None, 0, 16, None) == pa.PA_OK                  # nothing to read: no launch


def test_pack_rejects_malformed_sequences():
    dims = pa.make_dims(8, 16, 4, 2, 64)
    with pytest.raises(pa.PagedAttnError) as e:  # query longer than the sequence
        pa.pa_pack_prefill(dims, [10], [11], [[0]], pin=False)
    assert e.value.code == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PagedAttnError):  # too few blocks
        pa.pa_pack_prefill(dims, [33], [33], [[0, 1]], pin=False)
    with pytest.raises(pa.PagedAttnError):  # block id outside the pool
        pa.pa_pack_prefill(dims, [5], [5], [[8]], pin=False)
    with pytest.raises(pa.PagedAttnError):
        pa.pa_pack_decode(dims, [-1], [[0]], pin=False)
    with pytest.raises(pa.PagedAttnError):  # split not a multiple of 64
        pa.pa_pack_decode(dims, [5], [[0]], split_tokens=100, pin=False)


def _prefill_arrays(plan, b):
    m = plan.meta
    return (plan.host_array(m.off_cu_seqlens_q, b + 1), plan.host_array(m.off_cu_seqlens_k, b + 1),
            plan.host_array(m.off_block_tables, b * m.max_blocks_per_seq).reshape(b, m.max_blocks_per_seq),
            plan.host_array(m.off_slot_mapping, m.total_q), plan.host_array(m.off_tiles, 8 * m.num_tiles).reshape(-1, 8))


@pytest.mark.parametrize("name", ["tiny", "qwen3_prefix", "qwen3_chunked", "qwen3_prefill_128"])
def test_pack_prefill_matches_definitions(name):
    w = workloads.make(name)
    p = w.pool
    for batch in w.batches:
        if batch.kind != "prefill":
            continue
        dims = pa.make_dims(p.num_blocks, p.block_size, batch.num_heads, p.num_kv_heads, p.head_dim)
        plan = pa.pa_pack_prefill(dims, batch.seq_lens, batch.query_lens, batch.block_lists, pin=False)
        B = batch.num_seqs
        cu_q, cu_k, bt, slots, tiles = _prefill_arrays(plan, B)
        assert cu_q.tolist() == [0] + np.cumsum(batch.query_lens).tolist()
        assert cu_k.tolist() == [0] + np.cumsum(batch.seq_lens).tolist()
        # slots: bit-exact against the oracle's own slot mapping
        want = oracle.slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, p.block_size)
        assert np.array_equal(slots, want)
        for b in range(B):
            n = -(-int(batch.seq_lens[b]) // p.block_size)
            assert bt[b, :n].tolist() == batch.block_lists[b][:n].tolist()
            assert (bt[b, n:] == -1).all()
        # work items: each (seq, query row, kv head) exactly once, longest first;
        # one item = two query tiles of P positions
        G = batch.num_heads // p.num_kv_heads
        P = plan.meta.rows_per_tile
        assert P == 128 // G
        cover = {}
        for s, q0, g, nkt, cq, lq_, lk_, blk0 in tiles.tolist():
            lq, lk = int(batch.query_lens[s]), int(batch.seq_lens[s])
            assert (cq, lq_, lk_, blk0) == (int(cu_q[s]), lq, lk, int(batch.block_lists[s][0]))
            assert q0 % (2 * P) == 0
            last = min(q0 + 2 * P, lq) - 1
            assert nkt == -(-(lk - lq + last + 1) // 128)
            for i in range(q0, last + 1):
                cover[(s, i, g)] = cover.get((s, i, g), 0) + 1
        assert len(cover) == int(batch.query_lens.sum()) * p.num_kv_heads
        assert set(cover.values()) == {1}
        assert (np.diff(tiles[:, 3]) <= 0).all()


@pytest.mark.parametrize("split", [0, 64, 256, 1024])
def test_pack_decode_split_plan(split):
    w = workloads.qwen3_decode(num_seqs=32)
    p, batch = w.pool, w.batches[0]
    dims = pa.make_dims(p.num_blocks, p.block_size, batch.num_heads, p.num_kv_heads, p.head_dim)
    plan = pa.pa_pack_decode(dims, batch.seq_lens, batch.block_lists, split_tokens=split, pin=False)
    m = plan.meta
    B = batch.num_seqs
    slots = plan.host_array(m.off_slot_mapping, B)
    want = oracle.slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, p.block_size)
    assert np.array_equal(slots, want)
    assert np.array_equal(plan.host_array(m.off_context_lens, B), batch.seq_lens)
    items = plan.host_array(m.off_items, 4 * m.num_items).reshape(-1, 4)
    seq_items = plan.host_array(m.off_seq_items, B + 1)
    ranges = {}
    for s, k0, k1, slot in items.tolist():
        assert k0 % 64 == 0 and k1 > k0
        ranges.setdefault(s, []).append((k0, k1, slot))
    used = []
    for b in range(B):
        r = sorted(ranges[b])
        assert r[0][0] == 0 and r[-1][1] == batch.seq_lens[b]
        assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
        n = seq_items[b + 1] - seq_items[b]
        if len(r) == 1:
            assert n == 0 and r[0][2] == -1
        else:
            assert n == len(r)
            assert sorted(x[2] for x in r) == list(range(seq_items[b], seq_items[b + 1]))
            used += [x[2] for x in r]
    assert m.num_partials == seq_items[-1] == len(used)
    assert m.workspace_bytes >= m.num_partials * batch.num_heads * (p.head_dim + 1) * 4
    lens = items[:, 2] - items[:, 1]
    assert (np.diff(lens) <= 0).all()
    if split:
        assert m.split_tokens == split
        assert lens.max() <= split


def test_pack_decode_zero_context_is_an_empty_item():
    dims = pa.make_dims(8, 16, 4, 2, 64)
    plan = pa.pa_pack_decode(dims, [0, 20], [[], [3, 4]], split_tokens=64, pin=False)
    items = plan.host_array(plan.meta.off_items, 4 * plan.meta.num_items).reshape(-1, 4).tolist()
    assert [0, 0, 0, -1] in items
    assert plan.host_array(plan.meta.off_slot_mapping, 2).tolist() == [-1, 4 * 16 + 3]


def _fixed_plan(ctx, max_ctx, split, bs=16, seed=0):
    rng = np.random.default_rng(seed)
    nb = sum(-(-int(c) // bs) for c in ctx) + 3
    perm = rng.permutation(nb).astype(np.int32)
    blocks, o = [], 0
    for c in ctx:
        n = -(-int(c) // bs)
        blocks.append(perm[o:o + n])
        o += n
    dims = pa.make_dims(nb, bs, 8, 2, 128)
    return pa.pa_pack_decode_fixed(dims, ctx, blocks, max_ctx, split, pin=False), blocks, bs


META_SHAPE = ("num_seqs", "max_blocks_per_seq", "num_items", "split_tokens", "max_splits", "num_partials",
              "off_context_lens", "off_block_tables", "off_slot_mapping", "off_items", "off_seq_items",
              "total_bytes", "workspace_bytes")


@pytest.mark.parametrize("split", [0, 64, 256])
def test_pack_decode_fixed_shapes_do_not_depend_on_contexts(split):
    """Graph replay needs the same sizes and offsets for any contexts in the bucket."""
    metas = []
    for ctx in ([1000, 17, 0, 512], [1, 1024, 1024, 0], [0, 0, 0, 5], [64, 128, 192, 256]):
        plan, _, _ = _fixed_plan(np.array(ctx, np.int32), 1024, split)
        metas.append(tuple(getattr(plan.meta, f) for f in META_SHAPE))
    assert len(set(metas)) == 1
    S = -(-1024 // (split or 1024))
    assert metas[0][2] == 4 * S and metas[0][1] == 64


@pytest.mark.parametrize("split", [0, 64, 320])
def test_pack_decode_fixed_items(split):
    """Ranges tile [0, ctx) in order, empty ranges are (0, 0), exactly one range ends at ctx."""
    ctx = np.array([700, 1, 0, 640, 333, 1000], np.int32)
    plan, blocks, bs = _fixed_plan(ctx, 1000, split, seed=3)
    m = plan.meta
    items = plan.host_array(m.off_items, 4 * m.num_items).reshape(-1, 4)
    S = m.max_splits
    for b, c in enumerate(ctx):
        mine = items[b * S:(b + 1) * S]
        assert (mine[:, 0] == b).all()
        covered = [k for _, k0, k1, _ in mine for k in range(k0, k1)]
        assert covered == list(range(int(c)))
        assert sum(1 for _, k0, k1, _ in mine if k1 == c and k1 > k0) == (1 if c > 0 else 0)
        assert all((k0, k1) == (0, 0) for _, k0, k1, _ in mine if k1 <= k0)
        assert list(mine[:, 3]) == (list(range(b * S, (b + 1) * S)) if S > 1 else [-1] * S)
    slots = plan.host_array(m.off_slot_mapping, len(ctx))
    for b, c in enumerate(ctx):
        want = -1 if c == 0 else int(blocks[b][(c - 1) // bs]) * bs + (c - 1) % bs
        assert slots[b] == want


def test_pack_decode_fixed_rejects_contexts_over_the_bucket():
    ctx = np.array([10, 2000], np.int32)
    with pytest.raises(pa.PagedAttnError):
        _fixed_plan(ctx, 1024, 64)


def test_int8_fused_and_copy_calls_reject_bad_args_without_touching_the_gpu():
    """Host-side checks of the INT8, fused-decode and block-copy entry points (no launch on failure)."""
    dims = pa.make_dims(4, 16, 4, 2, 64)
    L = pa.lib()
    f = ctypes.c_float
    # quantising store: NULL scales, misaligned scales, zero tokens is a no-op
    assert L.pa_store_kvcache_int8(ctypes.byref(dims), 16, 16, 16, 16, None, 16, 16, 1, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache_int8(ctypes.byref(dims), 16, 16, 16, 16, 24, 16, 16, 1, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache_int8(ctypes.byref(dims), None, None, None, None, None, None, None, 0, None) == pa.PA_OK
    assert L.pa_store_kvcache_int8(ctypes.byref(dims), 16, 16, 16, 16, 16, 16, 16, -2, None) == pa.PA_ERR_INVALID_ARG
    # INT8 decode: NULL / misaligned scales, bad scale value, short workspace
    dm = pa.pa_decode_meta()
    dm.num_items, dm.num_seqs, dm.max_blocks_per_seq, dm.max_splits = 1, 1, 1, 1
    args = (ctypes.byref(dims), 16, 16, 16)
    assert L.pa_decode_int8(*args, None, 16, 16, 16, f(0.1), 16, ctypes.byref(dm), 16, 16, None, 0,
                            None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_int8(*args, 16, 40, 16, 16, f(0.1), 16, ctypes.byref(dm), 16, 16, None, 0,
                            None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_int8(*args, 16, 16, 16, 16, f(float("nan")), 16, ctypes.byref(dm), 16, 16, None, 0,
                            None) == pa.PA_ERR_INVALID_ARG
    dm.workspace_bytes = 512
    assert L.pa_decode_int8(*args, 16, 16, 16, 16, f(0.1), 16, ctypes.byref(dm), 16, 16, None, 0,
                            None) == pa.PA_ERR_WORKSPACE
    dm.workspace_bytes = 0
    # INT8 prefill: unsupported dims are rejected before anything else
    bad = pa.make_dims(4, 16, 4, 2, 96)
    pm = pa.pa_prefill_meta()
    pm.num_tiles, pm.total_q, pm.num_seqs, pm.max_blocks_per_seq, pm.rows_per_tile = 1, 1, 1, 1, 64
    pm.scratch_blocks, pm.scratch_pitch = 1, 1
    pm.workspace_bytes = 128 * 2 * 64 * 4  # dims: 2 KV heads, D 64

    def int8_call(d=dims, ks=16, stab=16, ws=16, ws_bytes=pm.workspace_bytes):
        return L.pa_prefill_varlen_int8(ctypes.byref(d), 16, 16, 16, ks, 16, 16, 16, 16, stab, 16, f(0.1), 16,
                                        ctypes.byref(pm), 16, ws, ws_bytes, None)

    assert int8_call(d=bad) == pa.PA_ERR_UNSUPPORTED
    assert int8_call(ks=None) == pa.PA_ERR_INVALID_ARG                      # scales
    assert int8_call(stab=None) == pa.PA_ERR_INVALID_ARG                    # scratch tables
    assert int8_call(ws=None) == pa.PA_ERR_INVALID_ARG                      # workspace
    assert int8_call(ws=24) == pa.PA_ERR_INVALID_ARG                        # misaligned workspace
    assert int8_call(ws_bytes=pm.workspace_bytes - 16) == pa.PA_ERR_WORKSPACE
    pm.workspace_bytes += 16  # not the scratch size of these dims
    assert int8_call(ws_bytes=1 << 30) == pa.PA_ERR_INVALID_ARG
    pm.workspace_bytes -= 16
    # fused decode: NULL new-token rows or slot mapping
    assert L.pa_decode_fused(ctypes.byref(dims), 16, None, 16, 16, 16, 16, 16, 16, f(0.1), 16, ctypes.byref(dm), 16,
                             16, None, 0, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_fused(ctypes.byref(dims), 16, 16, 16, 16, 16, None, 16, 16, f(0.1), 16, ctypes.byref(dm), 16,
                             16, None, 0, None) == pa.PA_ERR_INVALID_ARG
    # block copy: negative count, NULL triples, zero triples is a no-op
    assert L.pa_copy_blocks(ctypes.byref(dims), 16, 16, 16, -1, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_copy_blocks(ctypes.byref(dims), 16, 16, None, 2, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_copy_blocks(ctypes.byref(dims), None, None, None, 0, None) == pa.PA_OK
    # static-scratch decode: a plan larger than the library array is refused
    dm.workspace_bytes = pa.PA_DECODE_STATIC_SCRATCH_BYTES + 256
    assert L.pa_decode_static(ctypes.byref(dims), 16, 16, 16, 16, 16, f(0.1), 16, ctypes.byref(dm), 16, 16,
                              None) == pa.PA_ERR_WORKSPACE


def test_pack_prefill_prefix_aligned_flag():
    """meta.prefix_aligned: every cached prefix a multiple of min(block_size, 128)."""
    for bs, lens, qlens, expect in ((16, [40, 17], [8, 17], 1),       # prefixes 32, 0
                                    (16, [40, 17], [9, 17], 0),       # prefix 31
                                    (256, [300, 700], [44, 444], 1),  # prefixes 256, 256: boxes of 128
                                    (256, [300], [172], 1),           # prefix 128: half a block, 128-aligned
                                    (256, [300], [100], 0),           # prefix 200
                                    (32, [64], [64], 1),              # no prefix
                                    (16, [40, 17], [8, 0], 1)):       # prefix 17 but no new tokens
        dims = pa.make_dims(64, bs, 4, 2, 64)
        blocks = [list(range(i * 8, i * 8 + -(-n // bs))) for i, n in enumerate(lens)]
        plan = pa.pa_pack_prefill(dims, lens, qlens, blocks, pin=False)
        assert plan.meta.prefix_aligned == expect, (bs, lens, qlens)


def test_prefill_fused_rejects_bad_args_without_touching_the_gpu():
    dims = pa.make_dims(4, 16, 4, 2, 64)
    L = pa.lib()
    pm = pa.pa_prefill_meta()
    pm.num_tiles, pm.total_q, pm.num_seqs, pm.max_blocks_per_seq, pm.rows_per_tile = 1, 1, 1, 1, 64
    f = ctypes.c_float
    # NULL new-token rows, NULL slot mapping, misaligned rows, bad scale
    assert L.pa_prefill_varlen_fused(ctypes.byref(dims), 16, None, 16, 16, 16, 16, 16, 16, 16, f(0.1), 16,
                                     ctypes.byref(pm), 16, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_prefill_varlen_fused(ctypes.byref(dims), 16, 16, 16, 16, 16, 16, 16, 16, None, f(0.1), 16,
                                     ctypes.byref(pm), 16, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_prefill_varlen_fused(ctypes.byref(dims), 16, 24, 16, 16, 16, 16, 16, 16, 16, f(0.1), 16,
                                     ctypes.byref(pm), 16, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_prefill_varlen_fused(ctypes.byref(dims), 16, 16, 16, 16, 16, 16, 16, 16, 16, f(-1.0), 16,
                                     ctypes.byref(pm), 16, None) == pa.PA_ERR_INVALID_ARG
    pm.num_tiles = 0  # nothing to do: no launch, no error
    assert L.pa_prefill_varlen_fused(ctypes.byref(dims), None, None, None, None, None, None, None, None, None, f(0.1),
                                     None, ctypes.byref(pm), None, None) == pa.PA_OK


def test_prefill_int8_fused_rejects_bad_args_without_touching_the_gpu():
    dims = pa.make_dims(4, 16, 4, 2, 64)
    L = pa.lib()
    pm = pa.pa_prefill_meta()
    pm.num_tiles, pm.total_q, pm.num_seqs, pm.max_blocks_per_seq, pm.rows_per_tile = 1, 1, 1, 1, 64
    pm.scratch_blocks, pm.scratch_pitch, pm.workspace_bytes = 1, 1, 128 * 2 * 64 * 4
    f = ctypes.c_float

    def call(q=16, k=16, v=16, kc=16, vc=16, ks=16, vs=16, slots=16, scale=0.1, sseq=16, ws=16):
        return L.pa_prefill_varlen_int8_fused(ctypes.byref(dims), q, k, v, kc, vc, ks, vs, 16, 16, 16, slots, 16,
                                              sseq, f(scale), 16, ctypes.byref(pm), 16, ws, pm.workspace_bytes, None)

    assert call(k=None) == pa.PA_ERR_INVALID_ARG       # new-token rows
    assert call(vs=None) == pa.PA_ERR_INVALID_ARG      # scales
    assert call(slots=None) == pa.PA_ERR_INVALID_ARG   # slot mapping
    assert call(sseq=None) == pa.PA_ERR_INVALID_ARG    # the plan's scratch block owners
    assert call(ws=None) == pa.PA_ERR_INVALID_ARG      # workspace
    assert call(v=24) == pa.PA_ERR_INVALID_ARG         # misaligned rows
    assert call(ks=40) == pa.PA_ERR_INVALID_ARG        # misaligned scales
    assert call(scale=-1.0) == pa.PA_ERR_INVALID_ARG
    pm.num_tiles = 0  # nothing to do: no launch, no error
    assert L.pa_prefill_varlen_int8_fused(ctypes.byref(dims), None, None, None, None, None, None, None, None, None,
                                          None, None, None, None, f(0.1), None, ctypes.byref(pm), None, None, 0,
                                          None) == pa.PA_OK


def test_pack_prefill_scratch_tables():
    """The INT8 prefill's scratch cache: ceil(seq_len / 128) consecutive 128-token blocks for each
    sequence with new tokens, in sequence order (none for a sequence without new tokens), the tables
    -1 padded to the widest sequence, each scratch block's entry (sequence, first key, key count,
    cached prefix, packed row of its new keys minus the prefix), and K + V bf16 bytes."""
    dims = pa.make_dims(512, 16, 8, 2, 128)
    lens, qlens = [300, 17, 128, 129, 1000], [8, 0, 128, 1, 5]
    blocks, o = [], 0
    for n in lens:
        blocks.append(list(range(o, o + -(-n // 16))))
        o += -(-n // 16)
    plan = pa.pa_pack_prefill(dims, lens, qlens, blocks, pin=False)
    m = plan.meta
    per = [-(-n // 128) if q > 0 else 0 for n, q in zip(lens, qlens)]   # 3, 0, 1, 2, 8
    assert m.scratch_blocks == sum(per) == 14 and m.scratch_pitch == max(per) == 8
    assert m.workspace_bytes == 14 * 128 * 2 * 128 * 2 * 2
    tab = np.asarray(plan.host_array(m.off_scratch_tables, 5 * 8)).reshape(5, 8)
    first = np.concatenate([[0], np.cumsum(per)[:-1]])
    for b in range(5):
        want = [first[b] + i if i < per[b] else -1 for i in range(8)]
        assert list(tab[b]) == want, b
    items = np.asarray(plan.host_array(m.off_scratch_items, 14 * 8)).reshape(14, 8)
    cu_q = np.concatenate([[0], np.cumsum(qlens)])
    want = []
    for b in range(5):
        for i in range(per[b]):
            cached = lens[b] - qlens[b]
            want.append([b, 128 * i, lens[b], cached, cu_q[b] - cached, 0, 0, 0])
    assert items.tolist() == want
    assert [w[0] for w in want] == [0, 0, 0, 2, 3, 3] + [4] * 8
    assert m.off_scratch_tables >= m.off_tiles + 4 * 8 * m.num_tiles
    assert m.off_scratch_items >= m.off_scratch_tables + 4 * 5 * 8 and m.off_scratch_items % 16 == 0
    assert m.off_scratch_items + 4 * 8 * 14 <= m.total_bytes


def test_pack_prefill_scratch_without_new_tokens():
    """No sequence with new tokens: no scratch block, no workspace, tables all -1 (and no work)."""
    dims = pa.make_dims(64, 16, 4, 2, 64)
    plan = pa.pa_pack_prefill(dims, [40, 17], [0, 0], [[0, 1, 2], [3, 4]], pin=False)
    m = plan.meta
    assert (m.num_tiles, m.scratch_blocks, m.workspace_bytes, m.scratch_pitch) == (0, 0, 0, 1)
    assert list(plan.host_array(m.off_scratch_tables, 2)) == [-1, -1]
    # the INT8 prefill over such a plan launches nothing and needs no workspace
    L = pa.lib()
    f = ctypes.c_float
    assert L.pa_prefill_varlen_int8(ctypes.byref(dims), None, None, None, None, None, None, None, None, None, None,
                                    f(0.1), None, ctypes.byref(m), None, None, 0, None) == pa.PA_OK
