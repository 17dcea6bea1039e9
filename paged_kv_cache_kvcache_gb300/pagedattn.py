"""Thin ctypes binding of libpagedattn (include/pagedattn.h), same entry-point names.

Argument marshalling only: every step of the path (metadata packing, KV
scatter, prefill, decode) runs in the native library; torch provides device
memory, pinned host memory and streams.  There is no fallback: if the CUDA
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import _build

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = 0, 1, 2, 3, 4

EXPORTS = ("pa_pack_prefill", "pa_pack_decode", "pa_upload", "pa_store_kvcache", "pa_prefill_varlen",
           "pa_decode", "pa_decode_static", "pa_copy_blocks", "pa_store_kvcache_int8", "pa_decode_int8",
           "pa_prefill_varlen_int8", "pa_pack_decode_fixed", "pa_decode_fused", "pa_copy_blocks_int8",
           "pa_decode_int8_fused", "pa_prefill_varlen_fused", "pa_prefill_varlen_int8_fused",
           "pa_last_error_string", "pa_read_device_error", "pa_selftest_bounded_wait", "pa_stream_read",
           "pa_version")

PA_DECODE_STATIC_SCRATCH_BYTES = 16 << 20


class pa_dims(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class pa_prefill_meta(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_q", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
                ("max_seqlen_k", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_tiles", ctypes.c_int32), ("rows_per_tile", ctypes.c_int32), ("prefix_aligned", ctypes.c_int32),
                ("off_cu_seqlens_q", ctypes.c_uint64), ("off_cu_seqlens_k", ctypes.c_uint64),
                ("off_block_tables", ctypes.c_uint64), ("off_slot_mapping", ctypes.c_uint64),
                ("off_tiles", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
                ("off_scratch_tables", ctypes.c_uint64), ("off_scratch_items", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64), ("scratch_blocks", ctypes.c_int32),
                ("scratch_pitch", ctypes.c_int32)]


class pa_decode_meta(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_items", ctypes.c_int32), ("split_tokens", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("num_partials", ctypes.c_int32), ("off_context_lens", ctypes.c_uint64),
                ("off_block_tables", ctypes.c_uint64), ("off_slot_mapping", ctypes.c_uint64),
                ("off_items", ctypes.c_uint64), ("off_seq_items", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64), ("workspace_bytes", ctypes.c_uint64)]


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} failed with code {code}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libpagedattn (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            L.pa_pack_prefill.argtypes = [P, I32, P, P, P, P, P, SZ, P]
            L.pa_pack_decode.argtypes = [P, I32, P, P, P, I32, P, SZ, P]
            L.pa_pack_decode_fixed.argtypes = [P, I32, P, P, P, I32, I32, P, SZ, P]
            L.pa_decode_fused.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ, P]
            L.pa_upload.argtypes = [P, P, SZ, P]
            L.pa_store_kvcache.argtypes = [P, P, P, P, P, P, I32, P]
            L.pa_prefill_varlen.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P]
            L.pa_prefill_varlen_fused.argtypes = [P, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P]
            L.pa_decode.argtypes = [P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ, P]
            L.pa_decode_static.argtypes = [P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P]
            L.pa_copy_blocks.argtypes = [P, P, P, P, I32, P]
            L.pa_copy_blocks_int8.argtypes = [P, P, P, P, P, P, I32, P]
            L.pa_decode_int8_fused.argtypes = [P, P, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ,
                                               P]
            L.pa_store_kvcache_int8.argtypes = [P, P, P, P, P, P, P, P, I32, P]
            L.pa_decode_int8.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, SZ, P]
            L.pa_prefill_varlen_int8.argtypes = [P] * 11 + [ctypes.c_float] + [P] * 4 + [SZ, P]
            L.pa_prefill_varlen_int8_fused.argtypes = [P] * 14 + [ctypes.c_float] + [P] * 4 + [SZ, P]
            L.pa_last_error_string.argtypes = []
            L.pa_last_error_string.restype = ctypes.c_char_p
            L.pa_read_device_error.argtypes = [P, P]
            L.pa_selftest_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.c_int, P]
            L.pa_stream_read.argtypes = [P, SZ, P, P]
            L.pa_version.argtypes = []
            for name in EXPORTS:
                if name not in ("pa_last_error_string",):
                    getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc: int, fn: str):
    if rc != PA_OK:
        raise PagedAttnError(rc, fn, pa_last_error_string())


def pa_last_error_string() -> str:
    return lib().pa_last_error_string().decode(errors="replace")


def pa_version() -> int:
    return int(lib().pa_version())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() > 0 else None
    return int(t)


def make_dims(num_blocks: int, block_size: int, num_heads: int, num_kv_heads: int, head_dim: int) -> pa_dims:
    return pa_dims(num_blocks, block_size, num_heads, num_kv_heads, head_dim)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else None


def _flatten(block_lists) -> tuple:
    """Per-sequence block lists -> (offsets [B+1], flat ids); an (offsets, ids) pair passes through."""
    if isinstance(block_lists, tuple) and len(block_lists) == 2 and isinstance(block_lists[0], np.ndarray):
        return block_lists
    off = np.zeros(len(block_lists) + 1, dtype=np.int32)
    for i, b in enumerate(block_lists):
        off[i + 1] = off[i] + len(b)
    ids = (np.concatenate([np.asarray(b, np.int32) for b in block_lists]) if len(block_lists)
           else np.zeros(0, np.int32))
    return off, _i32(ids)


@dataclass
class _Plan:
    meta: ctypes.Structure
    host: torch.Tensor                 # pinned uint8 image
    dev: Optional[torch.Tensor] = None  # device copy

    def upload(self, device="cuda", stream=None) -> "_Plan":
        """One asynchronous host-to-device copy of the packed image (pa_upload)."""
        n = int(self.meta.total_bytes)
        if self.dev is None or self.dev.numel() < n:
            self.dev = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        _check(lib().pa_upload(_ptr(self.dev), _ptr(self.host), n, _stream(stream)), "pa_upload")
        return self

    def dptr(self, off: int) -> int:
        assert self.dev is not None, "upload the plan first"
        return self.dev.data_ptr() + int(off)

    def host_array(self, off: int, count: int) -> np.ndarray:
        """Read back a packed int32 array from the host image (tests/debugging)."""
        buf = self.host.numpy()
        return np.frombuffer(buf, dtype=np.int32, count=count, offset=int(off)).copy()


class PrefillPlan(_Plan):
    @property
    def slot_mapping(self) -> int:
        return self.dptr(self.meta.off_slot_mapping)


class DecodePlan(_Plan):
    @property
    def slot_mapping(self) -> int:
        return self.dptr(self.meta.off_slot_mapping)


def _pack(fn_name, meta, args, into, pin, cls):
    fn = getattr(lib(), fn_name)
    host = into.host if into is not None else None
    if host is None:
        _check(fn(*args, None, 0, ctypes.byref(meta)), fn_name)
        host = torch.empty(max(int(meta.total_bytes), 256), dtype=torch.uint8, pin_memory=pin)
    rc = fn(*args, _ptr(host), host.numel(), ctypes.byref(meta))
    if rc == PA_ERR_WORKSPACE:  # reused buffer too small: grow it
        host = torch.empty(int(meta.total_bytes), dtype=torch.uint8, pin_memory=pin)
        rc = fn(*args, _ptr(host), host.numel(), ctypes.byref(meta))
    _check(rc, fn_name)
    if into is not None:
        into.meta, into.host = meta, host
        return into
    return cls(meta, host)


def pa_pack_prefill(dims: pa_dims, seq_lens, query_lens, block_lists, pin: bool = True,
                    into: Optional["PrefillPlan"] = None) -> "PrefillPlan":
    """Pack cu_seqlens, block tables, slot mapping and the tile list on the CPU.

    ``into`` reuses an earlier plan's pinned buffer (the caller must make sure
    no copy from it is still in flight).
    """
    seq_lens, query_lens = _i32(seq_lens), _i32(query_lens)
    off, ids = _flatten(block_lists)
    args = (ctypes.byref(dims), len(seq_lens), _np_ptr(seq_lens), _np_ptr(query_lens), _np_ptr(off), _np_ptr(ids))
    return _pack("pa_pack_prefill", pa_prefill_meta(), args, into, pin, PrefillPlan)


def pa_pack_decode(dims: pa_dims, context_lens, block_lists, split_tokens: int = 0, pin: bool = True,
                   into: Optional["DecodePlan"] = None) -> "DecodePlan":
    """Pack context lens, block tables, slot mapping and the split plan on the CPU."""
    ctx = _i32(context_lens)
    off, ids = _flatten(block_lists)
    args = (ctypes.byref(dims), len(ctx), _np_ptr(ctx), _np_ptr(off), _np_ptr(ids), int(split_tokens))
    return _pack("pa_pack_decode", pa_decode_meta(), args, into, pin, DecodePlan)


def pa_pack_decode_fixed(dims: pa_dims, context_lens, block_lists, max_context: int, split_tokens: int = 0,
                         pin: bool = True, into: Optional["DecodePlan"] = None) -> "DecodePlan":
    """Decode plan whose shapes depend only on (dims, len(context_lens), max_context, split_tokens).

    Padding entries have context 0 and an empty block list.  With ``into`` the
    previous plan's pinned buffer (and, after ``upload``, its device buffer)
    is reused, so launches captured in a CUDA graph stay valid.
    """
    ctx = _i32(context_lens)
    off, ids = _flatten(block_lists)
    args = (ctypes.byref(dims), len(ctx), _np_ptr(ctx), _np_ptr(off), _np_ptr(ids), int(max_context),
            int(split_tokens))
    return _pack("pa_pack_decode_fixed", pa_decode_meta(), args, into, pin, DecodePlan)


def pa_upload(dev_dst, host_src, nbytes: int, stream=None):
    _check(lib().pa_upload(_ptr(dev_dst), _ptr(host_src), int(nbytes), _stream(stream)), "pa_upload")


def pa_store_kvcache(dims: pa_dims, k, v, k_cache, v_cache, slot_mapping, num_tokens: Optional[int] = None,
                     stream=None):
    n = int(k.shape[0]) if num_tokens is None else int(num_tokens)
    _check(lib().pa_store_kvcache(ctypes.byref(dims), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(slot_mapping), n, _stream(stream)), "pa_store_kvcache")


def pa_prefill_varlen(dims: pa_dims, q, k_cache, v_cache, plan: PrefillPlan, scale: float, out, stream=None):
    m = plan.meta
    _check(lib().pa_prefill_varlen(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   plan.dptr(m.off_cu_seqlens_q), plan.dptr(m.off_cu_seqlens_k),
                                   plan.dptr(m.off_block_tables), float(scale), _ptr(out), ctypes.byref(m),
                                   plan.dptr(m.off_tiles), _stream(stream)), "pa_prefill_varlen")


def pa_prefill_varlen_fused(dims: pa_dims, q, k, v, k_cache, v_cache, plan: PrefillPlan, scale: float, out,
                            stream=None):
    """pa_store_kvcache of the new tokens' k/v at the plan's slots + pa_prefill_varlen, in one launch."""
    m = plan.meta
    _check(lib().pa_prefill_varlen_fused(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                         plan.dptr(m.off_cu_seqlens_q), plan.dptr(m.off_cu_seqlens_k),
                                         plan.dptr(m.off_block_tables), plan.dptr(m.off_slot_mapping), float(scale),
                                         _ptr(out), ctypes.byref(m), plan.dptr(m.off_tiles), _stream(stream)),
           "pa_prefill_varlen_fused")


def decode_workspace(plan: DecodePlan, device="cuda") -> Optional[torch.Tensor]:
    n = int(plan.meta.workspace_bytes)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def pa_decode(dims: pa_dims, q, k_cache, v_cache, plan: DecodePlan, scale: float, out, workspace=None,
              stream=None):
    m = plan.meta
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_decode(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                           plan.dptr(m.off_context_lens), plan.dptr(m.off_block_tables), float(scale), _ptr(out),
                           ctypes.byref(m), plan.dptr(m.off_items), plan.dptr(m.off_seq_items), _ptr(workspace),
                           ws_bytes, _stream(stream)), "pa_decode")


def pa_decode_fused(dims: pa_dims, q, k, v, k_cache, v_cache, plan: DecodePlan, scale: float, out, workspace=None,
                    stream=None):
    """Store each sequence's new K/V row and decode, in one launch (pa_store_kvcache + pa_decode)."""
    m = plan.meta
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_decode_fused(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                 plan.dptr(m.off_slot_mapping), plan.dptr(m.off_context_lens),
                                 plan.dptr(m.off_block_tables), float(scale), _ptr(out), ctypes.byref(m),
                                 plan.dptr(m.off_items), plan.dptr(m.off_seq_items), _ptr(workspace), ws_bytes,
                                 _stream(stream)), "pa_decode_fused")


def pa_decode_static(dims: pa_dims, q, k_cache, v_cache, plan: DecodePlan, scale: float, out, stream=None):
    """pa_decode without a workspace, for callers that cannot allocate device memory.

    The library's own 16 MiB scratch array stands in for the workspace; every
    call on a device shares it, so calls must not overlap on the GPU.  The
    first call on a device does a one-time address lookup: make it before any
    stream capture.
    """
    m = plan.meta
    _check(lib().pa_decode_static(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  plan.dptr(m.off_context_lens), plan.dptr(m.off_block_tables), float(scale),
                                  _ptr(out), ctypes.byref(m), plan.dptr(m.off_items), plan.dptr(m.off_seq_items),
                                  _stream(stream)), "pa_decode_static")


def pa_copy_blocks(dims: pa_dims, k_cache, v_cache, triples, num_triples: Optional[int] = None, stream=None):
    """Copy the first n rows of block src to block dst (K and V) for each (src, dst, n) triple."""
    n = int(triples.shape[0]) if num_triples is None else int(num_triples)
    _check(lib().pa_copy_blocks(ctypes.byref(dims), _ptr(k_cache), _ptr(v_cache), _ptr(triples), n,
                                _stream(stream)), "pa_copy_blocks")


def int8_cache(dims: pa_dims, device="cuda"):
    """Allocate an empty INT8 cache: (k_codes, v_codes, k_scale, v_scale).

    Codes int8 [num_blocks, block_size, Hkv, D]; scales fp16 [num_blocks, Hkv, block_size].
    """
    shape = (dims.num_blocks, dims.block_size, dims.num_kv_heads, dims.head_dim)
    sshape = (dims.num_blocks, dims.num_kv_heads, dims.block_size)
    return (torch.zeros(shape, dtype=torch.int8, device=device), torch.zeros(shape, dtype=torch.int8, device=device),
            torch.zeros(sshape, dtype=torch.float16, device=device),
            torch.zeros(sshape, dtype=torch.float16, device=device))


def pa_store_kvcache_int8(dims: pa_dims, k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                          num_tokens: Optional[int] = None, stream=None):
    """Quantise each new token's K/V head vectors (bf16) into int8 codes + fp16 scales at its slot."""
    n = int(k.shape[0]) if num_tokens is None else int(num_tokens)
    _check(lib().pa_store_kvcache_int8(ctypes.byref(dims), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), n, _stream(stream)),
           "pa_store_kvcache_int8")


def prefill_workspace(plan: PrefillPlan, device="cuda") -> Optional[torch.Tensor]:
    """The INT8 prefill's workspace (its bf16 scratch cache) for this plan."""
    n = int(plan.meta.workspace_bytes)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def _call_workspace(plan: PrefillPlan, workspace, device, stream):
    """The caller's workspace, or one allocated for this call (kept from reuse until the
    call's stream has passed it)."""
    if workspace is None:
        workspace = prefill_workspace(plan, device)
        if workspace is not None and stream is not None:
            st = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))
            workspace.record_stream(st)
    return workspace


def pa_prefill_varlen_int8(dims: pa_dims, q, k_cache, v_cache, k_scale, v_scale, plan: PrefillPlan, scale: float,
                           out, workspace=None, stream=None):
    """pa_prefill_varlen over an INT8 cache (same plan as pa_prefill_varlen; workspace of
    plan.meta.workspace_bytes, allocated here when not given)."""
    m = plan.meta
    workspace = _call_workspace(plan, workspace, q.device, stream)
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_prefill_varlen_int8(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                        _ptr(v_scale), plan.dptr(m.off_cu_seqlens_q), plan.dptr(m.off_cu_seqlens_k),
                                        plan.dptr(m.off_block_tables), plan.dptr(m.off_scratch_tables),
                                        plan.dptr(m.off_scratch_items), float(scale), _ptr(out), ctypes.byref(m),
                                        plan.dptr(m.off_tiles), _ptr(workspace), ws_bytes, _stream(stream)),
           "pa_prefill_varlen_int8")


def pa_prefill_varlen_int8_fused(dims: pa_dims, q, k, v, k_cache, v_cache, k_scale, v_scale, plan: PrefillPlan,
                                 scale: float, out, workspace=None, stream=None):
    """pa_store_kvcache_int8 of the new tokens' k/v at the plan's slots + pa_prefill_varlen_int8, in one call."""
    m = plan.meta
    workspace = _call_workspace(plan, workspace, q.device, stream)
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_prefill_varlen_int8_fused(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache),
                                              _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                              plan.dptr(m.off_cu_seqlens_q), plan.dptr(m.off_cu_seqlens_k),
                                              plan.dptr(m.off_block_tables), plan.dptr(m.off_slot_mapping),
                                              plan.dptr(m.off_scratch_tables), plan.dptr(m.off_scratch_items),
                                              float(scale), _ptr(out), ctypes.byref(m), plan.dptr(m.off_tiles),
                                              _ptr(workspace), ws_bytes, _stream(stream)),
           "pa_prefill_varlen_int8_fused")


def pa_decode_int8_fused(dims: pa_dims, q, k, v, k_cache, v_cache, k_scale, v_scale, plan: DecodePlan,
                         scale: float, out, workspace=None, stream=None):
    """Quantising store of each sequence's new K/V row + INT8 decode, in one launch."""
    m = plan.meta
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_decode_int8_fused(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(k_scale), _ptr(v_scale), plan.dptr(m.off_slot_mapping),
                                      plan.dptr(m.off_context_lens), plan.dptr(m.off_block_tables), float(scale),
                                      _ptr(out), ctypes.byref(m), plan.dptr(m.off_items), plan.dptr(m.off_seq_items),
                                      _ptr(workspace), ws_bytes, _stream(stream)), "pa_decode_int8_fused")


def pa_decode_int8(dims: pa_dims, q, k_cache, v_cache, k_scale, v_scale, plan: DecodePlan, scale: float, out,
                   workspace=None, stream=None):
    """pa_decode over an INT8 cache (same plan and workspace as pa_decode)."""
    m = plan.meta
    ws_bytes = int(workspace.numel()) if isinstance(workspace, torch.Tensor) else 0
    _check(lib().pa_decode_int8(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                _ptr(v_scale), plan.dptr(m.off_context_lens), plan.dptr(m.off_block_tables),
                                float(scale), _ptr(out), ctypes.byref(m), plan.dptr(m.off_items),
                                plan.dptr(m.off_seq_items), _ptr(workspace), ws_bytes, _stream(stream)),
           "pa_decode_int8")


def pa_copy_blocks_int8(dims: pa_dims, k_cache, v_cache, k_scale, v_scale, triples,
                        num_triples: Optional[int] = None, stream=None):
    """pa_copy_blocks on an INT8 cache: codes and each KV head's scale run."""
    n = int(triples.shape[0]) if num_triples is None else int(num_triples)
    _check(lib().pa_copy_blocks_int8(ctypes.byref(dims), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(triples), n, _stream(stream)), "pa_copy_blocks_int8")


def pa_selftest_bounded_wait(timeout_us: int, arrive_first: bool = False, stream=None):
    """Run the library's bounded mbarrier wait on a barrier nothing completes (or, with
    arrive_first, one it completes itself); a timeout shows as bit 4 of pa_read_device_error."""
    _check(lib().pa_selftest_bounded_wait(ctypes.c_uint32(int(timeout_us)), 1 if arrive_first else 0, _stream(stream)),
           "pa_selftest_bounded_wait")


def pa_stream_read(src: torch.Tensor, sink: torch.Tensor, stream=None):
    """Read every byte of the device tensor `src` once (streaming loads): the read-only
    bandwidth that bounds the decode kernels.  `sink` is a 4-byte device tensor."""
    _check(lib().pa_stream_read(_ptr(src), src.numel() * src.element_size(), _ptr(sink), _stream(stream)),
           "pa_stream_read")


def pa_read_device_error(stream=None) -> int:
    code = ctypes.c_uint32(0)
    _check(lib().pa_read_device_error(ctypes.byref(code), _stream(stream)), "pa_read_device_error")
    return int(code.value)
