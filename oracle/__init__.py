"""CPU oracle for paged KV-cache attention (fp64).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the bench's CPU-baseline leg, never by the product library.  It shares
no code with the CUDA path; ``ref.c`` is compiled here with gcc.

Every function here follows a definition on the pages (see ``ref.c`` for the
per-step citations):
  * ``slot_mapping``   - slot of each new token (nano-vllm walkthrough, Step 5)
  * ``store_kvcache``  - bit copy of K/V rows into their slots, -1 skipped (Step 4)
  * ``copy_blocks``    - copy-on-write fork of a shared block's valid rows (vLLM/SGLang labs §4)
  * ``copy_blocks_int8`` - the same fork on an INT8 cache (codes and per-head scale runs)
  * ``gather_dense``   - block_table[pos // bs], pos % bs resolution (mini-infer §2.2-2.3)
  * ``paged_attention``- causal softmax(q K^T * scale) V, bottom-right aligned,
                         in double precision (KV-cache toy of the inference notes)
  * ``quantize_rows`` / ``store_kvcache_int8`` / ``paged_attention_int8`` - INT8 KV
                         cache: per-(token, KV head) symmetric codes and fp16
                         scales, attention on the dequantised cache (nano-vLLM Q&A, Q3;
                         decode reads code * scale exactly, prefill rounded to bf16)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ref.c into _build/liboracle.so (gcc, OpenMP)."""
    src = os.path.join(_HERE, "ref.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", src,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_slot_mapping.restype = ctypes.c_int64
            lib.oracle_slot_mapping.argtypes = [ctypes.c_int, P, P, P, P, ctypes.c_int, P]
            lib.oracle_store_kvcache.restype = None
            lib.oracle_store_kvcache.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_int64]
            lib.oracle_copy_blocks.restype = None
            lib.oracle_copy_blocks.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64]
            lib.oracle_copy_blocks_int8.restype = None
            lib.oracle_copy_blocks_int8.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int]
            lib.oracle_gather_dense_int8.restype = None
            lib.oracle_gather_dense_int8.argtypes = [P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, P]
            lib.oracle_gather_dense.restype = None
            lib.oracle_gather_dense.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
            lib.oracle_paged_attention.restype = ctypes.c_int64
            lib.oracle_paged_attention.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P, ctypes.c_int]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_quantize_rows.restype = None
            lib.oracle_quantize_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, P]
            lib.oracle_store_kvcache_int8.restype = None
            lib.oracle_store_kvcache_int8.argtypes = [P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int]
            lib.oracle_paged_attention_int8.restype = ctypes.c_int64
            lib.oracle_paged_attention_int8.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P, ctypes.c_int,
                                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, P,
                                                        P, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array of the raw bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def flatten_blocks(block_lists):
    """Per-sequence block lists -> (offsets [B+1], flat ids)."""
    off = np.zeros(len(block_lists) + 1, dtype=np.int32)
    for i, b in enumerate(block_lists):
        off[i + 1] = off[i] + len(b)
    ids = np.concatenate([np.asarray(b, np.int32) for b in block_lists]) if block_lists else np.zeros(0, np.int32)
    return off, _i32(ids)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def slot_mapping(seq_lens, query_lens, block_lists, block_size: int) -> np.ndarray:
    lib = _load()
    seq_lens, query_lens = _i32(seq_lens), _i32(query_lens)
    off, ids = flatten_blocks(block_lists)
    out = np.empty(int(query_lens.sum()), dtype=np.int32)
    n = lib.oracle_slot_mapping(len(seq_lens), _ptr(seq_lens), _ptr(query_lens), _ptr(off), _ptr(ids),
                                block_size, _ptr(out))
    if n < 0:
        raise ValueError("position outside the sequence's block list")
    return out


def store_kvcache(k_cache: np.ndarray, v_cache: np.ndarray, k, v, slots) -> None:
    """In place on uint16 numpy caches of shape [num_blocks, bs, Hkv, D]."""
    lib = _load()
    kb, vb, slots = _bits(k), _bits(v), _i32(slots)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    row = int(np.prod(k_cache.shape[2:]))
    assert kb.size == slots.size * row
    lib.oracle_store_kvcache(_ptr(k_cache), _ptr(v_cache), _ptr(kb), _ptr(vb), _ptr(slots), slots.size, row)


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, triples, block_size: int) -> None:
    """In place on uint16 caches [num_blocks, bs, Hkv, D]: (src, dst, n) row copies."""
    lib = _load()
    tr = np.ascontiguousarray(np.asarray(triples, dtype=np.int32).reshape(-1, 3))
    row = int(np.prod(k_cache.shape[2:]))
    lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(tr), tr.shape[0], block_size, row)


def copy_blocks_int8(k_cache: np.ndarray, v_cache: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray,
                     triples) -> None:
    """In place on an INT8 cache: codes [nb, bs, Hkv, D] int8, scales [nb, Hkv, bs] fp16 bits."""
    lib = _load()
    tr = np.ascontiguousarray(np.asarray(triples, dtype=np.int32).reshape(-1, 3))
    nb, bs, hkv, d = k_cache.shape
    assert k_scale.shape == (nb, hkv, bs)
    lib.oracle_copy_blocks_int8(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(tr), tr.shape[0],
                                bs, hkv, d)


def gather_dense(cache, length: int, blocks, block_size: int) -> np.ndarray:
    """Dense [length, Hkv, D] float64 rows of one sequence."""
    lib = _load()
    c = _bits(cache)
    hkv, d = c.shape[2], c.shape[3]
    blocks = _i32(blocks)
    out = np.empty((length, hkv, d), dtype=np.float64)
    lib.oracle_gather_dense(_ptr(c), length, _ptr(blocks), hkv, d, block_size, _ptr(out))
    return out


def paged_attention(q, k_cache, v_cache, seq_lens, query_lens, block_lists, block_size: int,
                    scale: float, row_select=None, num_threads: int = 0):
    """Causal paged attention in fp64.

    Returns (out [T, Hq, D] float64, pairs) where pairs is the number of
    (query row, head, key) scores computed.  Rows not selected by
    ``row_select`` (bool/uint8 [T]) are NaN.
    """
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    seq_lens, query_lens = _i32(seq_lens), _i32(query_lens)
    off, ids = flatten_blocks(block_lists)
    t, hq, d = qb.shape
    hkv = kb.shape[2]
    out = np.full((t, hq, d), np.nan, dtype=np.float64)
    sel = None
    if row_select is not None:
        sel = np.ascontiguousarray(np.asarray(row_select, dtype=np.uint8))
        assert sel.size == t
    pairs = lib.oracle_paged_attention(_ptr(qb), _ptr(kb), _ptr(vb), len(seq_lens), _ptr(seq_lens),
                                       _ptr(query_lens), _ptr(off), _ptr(ids), hq, hkv, d, block_size,
                                       float(scale), _ptr(sel) if sel is not None else None, _ptr(out),
                                       int(num_threads))
    if pairs < 0:
        raise ValueError("malformed paged-attention input")
    return out, int(pairs)


def run_batch(pool_k: np.ndarray, pool_v: np.ndarray, batch, block_size: int, row_select=None,
              num_threads: int = 0):
    """Store the batch's new K/V into the (uint16) pool copies, then attend.

    The two steps in the order the attention layer runs them: store, then
    attention (nano-vllm walkthrough, Step 4).  Mutates pool_k / pool_v.
    """
    slots = slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, block_size)
    store_kvcache(pool_k, pool_v, batch.k, batch.v, slots)
    return paged_attention(batch.q, pool_k, pool_v, batch.seq_lens, batch.query_lens, batch.block_lists,
                           block_size, batch.scale, row_select=row_select, num_threads=num_threads)


# ---------------------------------------------------------------- INT8 KV cache


def f32_to_f16(x: float) -> int:
    return int(_load().oracle_f32_to_f16(float(x)))


def f16_to_f32(h: int) -> float:
    return float(_load().oracle_f16_to_f32(int(h)))


def quantize_rows(x):
    """bf16 [..., D] -> (int8 codes [..., D], uint16 fp16-scale bits [...])."""
    lib = _load()
    xb = _bits(x)
    d = xb.shape[-1]
    rows = xb.size // d
    codes = np.empty(xb.shape, dtype=np.int8)
    scales = np.empty(xb.shape[:-1], dtype=np.uint16)
    lib.oracle_quantize_rows(_ptr(xb), rows, d, _ptr(codes), _ptr(scales))
    return codes, scales


def store_kvcache_int8(k_cache: np.ndarray, v_cache: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray,
                       k, v, slots) -> None:
    """In place: int8 caches [num_blocks, bs, Hkv, D], uint16 (fp16 bits) scales [num_blocks, Hkv, bs]."""
    lib = _load()
    kb, vb, slots = _bits(k), _bits(v), _i32(slots)
    bs, hkv, d = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    assert k_scale.shape == (k_cache.shape[0], hkv, bs)
    lib.oracle_store_kvcache_int8(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(kb),
                                  _ptr(vb), _ptr(slots), slots.size, hkv, d, bs)


def paged_attention_int8(q, k_cache, v_cache, k_scale, v_scale, seq_lens, query_lens, block_lists,
                         block_size: int, scale: float, row_select=None, num_threads: int = 0,
                         values: str = "exact"):
    """Causal paged attention over an INT8 cache in fp64, the cached values read as
    code * fp16 scale: exactly (values="exact", the page's decode path) or rounded to bf16
    (values="bf16", the page's prefill path, which casts them to the model's dtype)."""
    assert values in ("exact", "bf16")
    lib = _load()
    qb = _bits(q)
    seq_lens, query_lens = _i32(seq_lens), _i32(query_lens)
    off, ids = flatten_blocks(block_lists)
    t, hq, d = qb.shape
    hkv = k_cache.shape[2]
    out = np.full((t, hq, d), np.nan, dtype=np.float64)
    sel = None
    if row_select is not None:
        sel = np.ascontiguousarray(np.asarray(row_select, dtype=np.uint8))
    pairs = lib.oracle_paged_attention_int8(_ptr(qb), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                            1 if values == "bf16" else 0, len(seq_lens), _ptr(seq_lens), _ptr(query_lens), _ptr(off), _ptr(ids),
                                            hq, hkv, d, block_size, float(scale),
                                            _ptr(sel) if sel is not None else None, _ptr(out), int(num_threads))
    if pairs < 0:
        raise ValueError("malformed paged-attention input")
    return out, int(pairs)


def run_batch_int8(k_cache, v_cache, k_scale, v_scale, batch, block_size: int, row_select=None):
    """Quantising store of the batch's new K/V, then attention on the INT8 cache (mutates the
    caches); a prefill batch reads the values rounded to bf16, a decode batch exactly."""
    slots = slot_mapping(batch.seq_lens, batch.query_lens, batch.block_lists, block_size)
    store_kvcache_int8(k_cache, v_cache, k_scale, v_scale, batch.k, batch.v, slots)
    return paged_attention_int8(batch.q, k_cache, v_cache, k_scale, v_scale, batch.seq_lens, batch.query_lens,
                                batch.block_lists, block_size, batch.scale, row_select=row_select,
                                values="bf16" if batch.kind == "prefill" else "exact")


def gather_dense_int8(codes, scales, length: int, blocks, block_size: int, values: str = "exact") -> np.ndarray:
    """Dense [length, Hkv, D] float64 values of one sequence of an INT8 cache (codes int8
    [nb, bs, Hkv, D], scales fp16 bits [nb, Hkv, bs]), exact or rounded to bf16."""
    assert values in ("exact", "bf16")
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.int8)
    sc = np.ascontiguousarray(scales, dtype=np.uint16)
    hkv, d = c.shape[2], c.shape[3]
    blocks = _i32(blocks)
    out = np.empty((length, hkv, d), dtype=np.float64)
    lib.oracle_gather_dense_int8(_ptr(c), _ptr(sc), length, _ptr(blocks), hkv, d, block_size,
                                 1 if values == "bf16" else 0, _ptr(out))
    return out
