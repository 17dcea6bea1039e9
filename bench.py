#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention hot path on one GB300.

One step = the whole path over one batch of seeded synthetic input:
  1. host metadata packing (pa_pack_prefill / pa_pack_decode) + one upload each,
     on a copy stream while the previous step computes (double-buffered images),
  2. KV scatter of the 4 x 4096 prompt tokens + causal varlen prefill, by default
     as one pa_prefill_varlen_fused launch (--prefill-path store+prefill: two),
  3. KV scatter of the 64 decode tokens + split-KV decode + LSE combine,
on the long-context Qwen2.5-7B attention shapes (28 q / 4 KV heads, head_dim
128, block 16): prefill 4 x 4096, decode 64 sequences at context 32768 through
fully permuted block tables.  Inputs are resident in HBM when timing starts;
the decode phase streams 4.3 GB of K/V per step, more than the 129 MB L2, so
every step starts with a cold L2.

Prints ONE JSON line.  value = prefill attention TFLOP/s (causal FLOPs
4*D*Hq*pairs over the prefill phase's device time); the decode KV-read GB/s
sits beside it under "decode".  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV-read GB/s (% of GB300 roofline), 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
# DRAM read + write bytes per launch from ncu captures of the current kernels on
# this workload: the prefill launch exactly as benched; the decode kernel on 16
# of the 64 sequences, scaled by 4 (traffic grows with the sequences).  Must be
# re-captured (or set to None) whenever one of these kernels changes.
NCU_TRAFFIC = {"qwen25": {"prefill": 232.9e6, "decode": 4.334e9}}
NCU_TRAFFIC_INT8 = {"qwen25": {"prefill": 249.7e6, "decode": 2.214e9}}  # prefill: gather + prefill kernel
NCU_TRAFFIC_FUSED_PREFILL = {"qwen25": 268.8e6}
NCU_TRAFFIC_INT8_FUSED_PREFILL = {"qwen25": 267.5e6}  # quantising gather + prefill kernel
NCU_TRAFFIC_COPY_BLOCKS = 488.3e6  # 268.5 MB read + 219.7 MB written (part of the writes still in L2 at exit)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["qwen25", "qwen3", "qwen3_prefill_32", "qwen3_prefill_128",
                                           "qwen3_prefix", "qwen3_chunked"], default="qwen25",
                    help="qwen25: the long-context case (default); the others pair a Qwen3-0.6B prefill "
                         "batch with the 256-sequence Qwen3 decode batch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--phase", choices=["both", "prefill", "decode"], default="both",
                    help="run only one phase (small profiling cases); the JSON line needs both")
    ap.add_argument("--decode-seqs", type=int, default=64, help="decode batch (64 = the full workload)")
    ap.add_argument("--kv", choices=["bf16", "int8"], default="bf16",
                    help="cache format: bf16, or int8 codes + fp16 scales (quantising store, fused-dequant "
                         "prefill and decode)")
    ap.add_argument("--prefill-path", choices=["store+prefill", "fused"], default="fused",
                    help="prompt batch: store + prefill (two launches), or the fused call "
                         "(pa_prefill_varlen_fused; INT8: pa_prefill_varlen_int8_fused)")
    ap.add_argument("--decode-path", choices=["store+decode", "fused", "mixed"], default="store+decode",
                    help="fused: store and decode in one launch (pa_decode_fused / pa_decode_int8_fused); "
                         "mixed (bf16): the decode rows join the prefill rows as Lq = 1 varlen rows of one "
                         "pa_prefill_varlen launch over one pool, timed against the separate launches")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- ranks


def max_over_ranks(value: float) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workload


def make_workload(name, device, decode_seqs=64):
    from paged_kv_cache_kvcache_gb300 import workloads
    if name == "qwen25":
        return workloads.make("qwen25_prefill", device), workloads.qwen25_decode(device, num_seqs=decode_seqs), \
            f"qwen25_long: prefill 4x4096 + decode {decode_seqs}x32768, Hq 28 / Hkv 4, D 128, block 16, permuted pools"
    pre = {"qwen3": "qwen3_prefill_256"}.get(name, name)
    desc = {"qwen3_prefill_256": "prefill 8x256", "qwen3_prefill_32": "prefill 8x32",
            "qwen3_prefill_128": "prefill 8x128", "qwen3_prefix": "prefix-cache prefill 8x(44 of 300, block 0 shared)",
            "qwen3_chunked": "chunked prefill 16x(prefix U{0..1024} + chunk U{1..512})"}[pre]
    return workloads.make(pre, device), workloads.make("qwen3_decode", device), \
        f"{name}: {desc} + decode 256 x ctx(in+out, in/out~U{{100..1024}}), Hq 16 / Hkv 8, D 128, block 256"


def prefill_flops(batch) -> float:
    lk = batch.seq_lens.astype(np.int64)
    lq = batch.query_lens.astype(np.int64)
    pairs = int(np.sum(lq * (lk - lq) + lq * (lq + 1) // 2))
    return 4.0 * batch.q.shape[2] * batch.num_heads * pairs


def decode_bytes(batch, pool, kv_fmt="bf16") -> float:
    ctx = batch.seq_lens.astype(np.int64)
    # K and V per key and KV head: D bf16 values, or D int8 codes + one fp16 scale
    per = pool.head_dim * 2 if kv_fmt == "bf16" else pool.head_dim + 2
    kv = float(np.sum(ctx)) * pool.num_kv_heads * per * 2
    qo = 2.0 * batch.q.numel() * 2
    tables = float(np.sum(-(-ctx // pool.block_size))) * 4 + ctx.size * 4
    return kv + qo + tables


def store_bytes(batch) -> float:
    return 2.0 * 2 * batch.k.numel() * 2  # K and V, read + write


def mixed_batch(wp, wd):
    """One pool (prefill blocks, then decode blocks) and one varlen batch: the prefill
    sequences followed by the decode sequences as query-length-1 rows."""
    from paged_kv_cache_kvcache_gb300 import workloads
    bp, bd, pp, pd = wp.batches[0], wd.batches[0], wp.pool, wd.pool
    assert (pp.block_size, pp.num_kv_heads, pp.head_dim, bp.num_heads) == \
        (pd.block_size, pd.num_kv_heads, pd.head_dim, bd.num_heads), "mixed: the two phases need one cache shape"
    kc = torch.cat([pp.k_cache, pd.k_cache])
    vc = torch.cat([pp.v_cache, pd.v_cache])
    lists = list(bp.block_lists) + [np.asarray(b, np.int32) + pp.num_blocks for b in bd.block_lists]
    b = workloads.Batch("prefill", np.concatenate([bp.seq_lens, bd.seq_lens]).astype(np.int32),
                        np.concatenate([bp.query_lens, np.ones(len(bd.seq_lens), np.int32)]).astype(np.int32),
                        lists, torch.cat([bp.q, bd.q]), torch.cat([bp.k, bd.k]), torch.cat([bp.v, bd.v]),
                        bp.num_heads, bp.scale)
    return kc, vc, b


class Step:
    """Device-resident state of one replica and the calls of one step."""

    def __init__(self, wp, wd, stream, kv="bf16", fused=False, mixed=False, prefill_fused=False):
        from paged_kv_cache_kvcache_gb300 import pagedattn as pa
        self.pa = pa
        self.s = stream
        self.int8, self.fused, self.mixed = kv == "int8", fused, mixed
        self.prefill_fused = prefill_fused and not mixed
        self.wp, self.wd = wp, wd
        self.bp, self.bd = wp.batches[0], wd.batches[0]
        pp, pd = wp.pool, wd.pool
        self.dims_p = pa.make_dims(pp.num_blocks, pp.block_size, self.bp.num_heads, pp.num_kv_heads, pp.head_dim)
        self.dims_d = pa.make_dims(pd.num_blocks, pd.block_size, self.bd.num_heads, pd.num_kv_heads, pd.head_dim)
        self.kc_p, self.vc_p = pp.k_cache, pp.v_cache
        self.kc_d, self.vc_d = pd.k_cache, pd.v_cache
        self.blocks_p = pa._flatten(self.bp.block_lists)
        self.blocks_d = pa._flatten(self.bd.block_lists)
        self.out_p = torch.empty_like(self.bp.q)
        self.out_d = torch.empty_like(self.bd.q)
        # double-buffered pinned metadata images (no write-after-read hazard with in-flight copies)
        self.plans_p = [pa.pa_pack_prefill(self.dims_p, self.bp.seq_lens, self.bp.query_lens, self.blocks_p)
                        .upload(stream=stream) for _ in range(2)]
        self.plans_d = [pa.pa_pack_decode(self.dims_d, self.bd.seq_lens, self.blocks_d).upload(stream=stream)
                        for _ in range(2)]
        self.up_ev = [torch.cuda.Event(), torch.cuda.Event()]
        for e in self.up_ev:
            e.record(stream)
        # run(): each step's metadata is packed and uploaded on a copy stream while the
        # previous step computes; plan_free[k] marks the last kernel that read slot k's images
        self.cs = torch.cuda.Stream(device=stream.device)
        self.plan_free = [torch.cuda.Event(), torch.cuda.Event()]
        for e in self.plan_free:
            e.record(stream)
        self.staged = [False, False]
        self.ws = pa.decode_workspace(self.plans_d[0])
        self.pipe_ev = {"p": [torch.cuda.Event(), torch.cuda.Event()], "d": [torch.cuda.Event(), torch.cuda.Event()]}
        for evs_ in self.pipe_ev.values():
            for e in evs_:
                e.record(stream)
        self.i = 0
        self.launches_per_step = 4 + (1 if self.plans_d[0].meta.num_partials > 0 else 0) - (1 if fused else 0)
        if self.prefill_fused:  # store and prefill in one launch
            self.launches_per_step -= 1
        if mixed:  # one launch for both phases' rows, over one pool
            self.kc_m, self.vc_m, self.bm = mixed_batch(wp, wd)
            self.dims_m = pa.make_dims(self.kc_m.shape[0], pp.block_size, self.bm.num_heads, pp.num_kv_heads,
                                       pp.head_dim)
            self.blocks_m = pa._flatten(self.bm.block_lists)
            self.out_m = torch.empty_like(self.bm.q)
            self.plans_m = [pa.pa_pack_prefill(self.dims_m, self.bm.seq_lens, self.bm.query_lens, self.blocks_m)
                            .upload(stream=stream) for _ in range(2)]
            self.launches_per_step = 2
        if self.int8:  # INT8 caches: the bf16 pools quantised once, every slot, by the library's store
            self.ws_p = pa.prefill_workspace(self.plans_p[0])  # the INT8 prefill's bf16 scratch cache
            self.c8_p = self._quantised(self.dims_p, pp)
            self.c8_d = self._quantised(self.dims_d, pd)
            torch.cuda.current_stream().synchronize()

    def _quantised(self, dims, pool):
        pa = self.pa
        n = pool.num_blocks * pool.block_size
        cache = pa.int8_cache(dims, pool.k_cache.device)
        slots = torch.arange(n, dtype=torch.int32, device=pool.k_cache.device)
        pa.pa_store_kvcache_int8(dims, pool.k_cache.view(n, pool.num_kv_heads, pool.head_dim),
                                 pool.v_cache.view(n, pool.num_kv_heads, pool.head_dim), *cache, slots, n,
                                 stream=self.s)
        return cache

    # ---- pipelined end-to-end steps: one phase's compute on explicit device buffers
    def prefill_on(self, q, k, v, out, slot):
        """Pack + upload + store + prefill of the prompt batch, reading q/k/v and writing out."""
        pa, s = self.pa, self.s
        self.pipe_ev["p"][slot].synchronize()  # the pinned plan image of this slot is free again
        plan = pa.pa_pack_prefill(self.dims_p, self.bp.seq_lens, self.bp.query_lens, self.blocks_p,
                                  into=self.plans_p[slot]).upload(stream=s)
        self.pipe_ev["p"][slot].record(s)
        if self.int8 and self.prefill_fused:
            pa.pa_prefill_varlen_int8_fused(self.dims_p, q, k, v, *self.c8_p, plan, self.bp.scale, out, self.ws_p,
                                            stream=s)
        elif self.int8:
            pa.pa_store_kvcache_int8(self.dims_p, k, v, *self.c8_p, plan.slot_mapping, self.bp.num_tokens, stream=s)
            pa.pa_prefill_varlen_int8(self.dims_p, q, *self.c8_p, plan, self.bp.scale, out, self.ws_p, stream=s)
        elif self.prefill_fused:
            pa.pa_prefill_varlen_fused(self.dims_p, q, k, v, self.kc_p, self.vc_p, plan, self.bp.scale, out, stream=s)
        else:
            pa.pa_store_kvcache(self.dims_p, k, v, self.kc_p, self.vc_p, plan.slot_mapping, self.bp.num_tokens,
                                stream=s)
            pa.pa_prefill_varlen(self.dims_p, q, self.kc_p, self.vc_p, plan, self.bp.scale, out, stream=s)

    def decode_on(self, q, k, v, out, slot):
        """Pack + upload + store + decode of the decode batch, reading q/k/v and writing out."""
        pa, s = self.pa, self.s
        self.pipe_ev["d"][slot].synchronize()
        plan = pa.pa_pack_decode(self.dims_d, self.bd.seq_lens, self.blocks_d, into=self.plans_d[slot]).upload(stream=s)
        self.pipe_ev["d"][slot].record(s)
        if self.int8 and self.fused:
            pa.pa_decode_int8_fused(self.dims_d, q, k, v, *self.c8_d, plan, self.bd.scale, out, self.ws, stream=s)
        elif self.int8:
            pa.pa_store_kvcache_int8(self.dims_d, k, v, *self.c8_d, plan.slot_mapping, self.bd.num_tokens, stream=s)
            pa.pa_decode_int8(self.dims_d, q, *self.c8_d, plan, self.bd.scale, out, self.ws, stream=s)
        elif self.fused:
            pa.pa_decode_fused(self.dims_d, q, k, v, self.kc_d, self.vc_d, plan, self.bd.scale, out, self.ws,
                               stream=s)
        else:
            pa.pa_store_kvcache(self.dims_d, k, v, self.kc_d, self.vc_d, plan.slot_mapping, self.bd.num_tokens,
                                stream=s)
            pa.pa_decode(self.dims_d, q, self.kc_d, self.vc_d, plan, self.bd.scale, out, self.ws, stream=s)

    def _stage(self, k, phase):
        """Pack slot k's metadata images on the host and upload them on the copy stream."""
        pa = self.pa
        self.up_ev[k].synchronize()  # the pinned images of slot k are free (their last upload is done)
        if self.mixed:
            plans = [pa.pa_pack_prefill(self.dims_m, self.bm.seq_lens, self.bm.query_lens, self.blocks_m,
                                        into=self.plans_m[k])]
        else:
            plans = []
            if phase != "decode":
                plans.append(pa.pa_pack_prefill(self.dims_p, self.bp.seq_lens, self.bp.query_lens, self.blocks_p,
                                                into=self.plans_p[k]))
            if phase != "prefill":
                plans.append(pa.pa_pack_decode(self.dims_d, self.bd.seq_lens, self.blocks_d, into=self.plans_d[k]))
        self.cs.wait_event(self.plan_free[k])  # no kernel still reads slot k's device images
        for plan in plans:
            plan.upload(stream=self.cs)
        self.up_ev[k].record(self.cs)
        self.staged[k] = True

    def run(self, ev=None, phase="both"):
        """Enqueue one step; ev = dict of event pairs for per-phase timing.

        The step's metadata (pack + upload) was staged on the copy stream while the
        previous step computed; the compute stream waits for it inside the prefill
        phase (so an upload that is late shows in the phase's time).
        """
        pa, s = self.pa, self.s
        k = self.i & 1
        self.i += 1
        if not self.staged[k]:
            self._stage(k, phase)
        self.staged[k] = False
        rec = (lambda name: ev[name].record(s)) if ev is not None else (lambda name: None)
        # ---- prefill phase
        rec("p0")
        s.wait_event(self.up_ev[k])
        if self.mixed:  # both phases' rows: one store, one prefill launch; the decode phase stays empty
            plan_m = self.plans_m[k]
            pa.pa_store_kvcache(self.dims_m, self.bm.k, self.bm.v, self.kc_m, self.vc_m, plan_m.slot_mapping,
                                self.bm.num_tokens, stream=s)
            rec("pk0")
            pa.pa_prefill_varlen(self.dims_m, self.bm.q, self.kc_m, self.vc_m, plan_m, self.bm.scale, self.out_m,
                                 stream=s)
            for n in ("pk1", "p1", "dk0", "dk1", "d1"):
                rec(n)
            self.plan_free[k].record(s)
            self._stage(1 - k, phase)
            return
        if phase == "decode":
            for n in ("pk0", "pk1", "p1"):
                rec(n)
            self._decode(ev, k, rec)
            self.plan_free[k].record(s)
            self._stage(1 - k, phase)
            return
        plan_p = self.plans_p[k]
        if self.int8 and self.prefill_fused:  # quantising store + gather, then the prefill
            rec("pk0")
            pa.pa_prefill_varlen_int8_fused(self.dims_p, self.bp.q, self.bp.k, self.bp.v, *self.c8_p, plan_p,
                                            self.bp.scale, self.out_p, self.ws_p, stream=s)
        elif self.int8:
            pa.pa_store_kvcache_int8(self.dims_p, self.bp.k, self.bp.v, *self.c8_p, plan_p.slot_mapping,
                                     self.bp.num_tokens, stream=s)
            rec("pk0")
            pa.pa_prefill_varlen_int8(self.dims_p, self.bp.q, *self.c8_p, plan_p, self.bp.scale, self.out_p,
                                      self.ws_p, stream=s)
        elif self.prefill_fused:  # store + prefill in one launch: the kernel time includes the store
            rec("pk0")
            pa.pa_prefill_varlen_fused(self.dims_p, self.bp.q, self.bp.k, self.bp.v, self.kc_p, self.vc_p, plan_p,
                                       self.bp.scale, self.out_p, stream=s)
        else:
            pa.pa_store_kvcache(self.dims_p, self.bp.k, self.bp.v, self.kc_p, self.vc_p, plan_p.slot_mapping,
                                self.bp.num_tokens, stream=s)
            rec("pk0")
            pa.pa_prefill_varlen(self.dims_p, self.bp.q, self.kc_p, self.vc_p, plan_p, self.bp.scale, self.out_p,
                                 stream=s)
        rec("pk1")
        rec("p1")
        if phase == "prefill":
            for n in ("dk0", "dk1", "d1"):
                rec(n)
        else:
            self._decode(ev, k, rec)
        self.plan_free[k].record(s)
        self._stage(1 - k, phase)

    def _decode(self, ev, k, rec):
        pa, s = self.pa, self.s
        # ---- decode phase (its metadata image was uploaded with the prefill's)
        plan_d = self.plans_d[k]
        if self.int8 and self.fused:  # quantising store + INT8 decode in one launch
            rec("dk0")
            pa.pa_decode_int8_fused(self.dims_d, self.bd.q, self.bd.k, self.bd.v, *self.c8_d, plan_d, self.bd.scale,
                                    self.out_d, self.ws, stream=s)
        elif self.int8:
            pa.pa_store_kvcache_int8(self.dims_d, self.bd.k, self.bd.v, *self.c8_d, plan_d.slot_mapping,
                                     self.bd.num_tokens, stream=s)
            rec("dk0")
            pa.pa_decode_int8(self.dims_d, self.bd.q, *self.c8_d, plan_d, self.bd.scale, self.out_d, self.ws, stream=s)
        elif self.fused:  # store + decode in one launch: the phase's kernel time includes the store
            rec("dk0")
            pa.pa_decode_fused(self.dims_d, self.bd.q, self.bd.k, self.bd.v, self.kc_d, self.vc_d, plan_d,
                               self.bd.scale, self.out_d, self.ws, stream=s)
        else:
            pa.pa_store_kvcache(self.dims_d, self.bd.k, self.bd.v, self.kc_d, self.vc_d, plan_d.slot_mapping,
                                self.bd.num_tokens, stream=s)
            rec("dk0")
            pa.pa_decode(self.dims_d, self.bd.q, self.kc_d, self.vc_d, plan_d, self.bd.scale, self.out_d, self.ws,
                         stream=s)
        rec("dk1")
        rec("d1")


def pipelined_e2e(step, phase, steps, warmup):
    """One phase end to end through the public API, copies overlapped across steps: while
    step i computes on the compute stream, step i+1's inputs are copied in from pinned host
    memory and step i-1's output is copied back out (one copy stream per direction, two
    device slots; events keep every copy off the buffers a step still uses).  Every timed
    step still moves all of its inputs in and its whole output out.
    Returns (ms per step, H2D bytes per step, D2H bytes per step)."""
    s = step.s
    b = step.bp if phase == "p" else step.bd
    run = step.prefill_on if phase == "p" else step.decode_on
    out0 = step.out_p if phase == "p" else step.out_d
    host_in = [t.cpu().pin_memory() for t in (b.q, b.k, b.v)]
    host_out = [torch.empty_like(out0, device="cpu").pin_memory() for _ in range(2)]
    dev = [[b.q, b.k, b.v, out0], [torch.empty_like(b.q), torch.empty_like(b.k), torch.empty_like(b.v),
                                   torch.empty_like(out0)]]
    ci, co = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    out_read = [torch.cuda.Event(), torch.cuda.Event()]
    used = [False, False]

    def one(i):
        k = i & 1
        q, kk, vv, out = dev[k]
        with torch.cuda.stream(ci):
            if used[k]:
                ci.wait_event(done[k])  # step i-2 has finished reading this slot's inputs
            q.copy_(host_in[0], non_blocking=True)
            kk.copy_(host_in[1], non_blocking=True)
            vv.copy_(host_in[2], non_blocking=True)
            in_ready[k].record(ci)
        s.wait_event(in_ready[k])
        if used[k]:
            s.wait_event(out_read[k])  # step i-2's output has left this slot
        run(q, kk, vv, out, k)
        done[k].record(s)
        with torch.cuda.stream(co):
            co.wait_event(done[k])
            host_out[k].copy_(out, non_blocking=True)
            out_read[k].record(co)
        used[k] = True

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(ci)
    for i in range(warmup, warmup + steps):
        one(i)
    t1.record(co)  # after the last output copy, which follows every earlier copy and step
    torch.cuda.synchronize()
    h2d = sum(int(t.numel() * t.element_size()) for t in host_in)
    d2h = int(host_out[0].numel() * host_out[0].element_size())
    return t0.elapsed_time(t1) / steps, h2d, d2h


class Clocks:
    """nvidia-smi sampling during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.proc = None
        self.index = index
        if not enabled:
            return
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0=None, t1=None):
        """Summarise samples taken in the wall-clock window [t0, t1] (widened to 0.5 s if it holds none)."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = [l.split(",") for l in open(self.f.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.f.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + r[0].split(".")[1]) if "." in r[0] else 0.0
                parsed.append((ts, float(r[2]), float(r[3]), r[6:10]))
            except (ValueError, IndexError):
                continue
        if not parsed:
            return None
        window = "timed region"
        sel = [x for x in parsed if t0 is None or (t0 <= x[0] <= t1)]
        if not sel:
            window = "timed region +/- 0.5 s"
            sel = [x for x in parsed if t0 - 0.5 <= x[0] <= t1 + 0.5] or parsed
        reasons = set()
        for x in sel:
            for n, v in zip(names, x[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [x[1] for x in sel]
        mx = sel[-1][2]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


# ---------------------------------------------------------------- CPU oracle legs


def copy_blocks_roofline(device, stream, hbm_peak, peak_src, iters=20, warmup=3):
    """Copy-on-write block copies (row f4) against the HBM roofline.

    8192 full-block copies (Qwen2.5 layout: block 16, 4 KV heads, D 128) between two
    halves of a scratch pool of 16384 blocks, src and dst permuted: 256 MB read and
    256 MB written per launch, so no launch is served from L2.  Work = bytes read +
    bytes written, like the copy-bandwidth peak it is compared with.
    """
    from paged_kv_cache_kvcache_gb300 import pagedattn as pa
    nb, bs, hkv, d, n = 16384, 16, 4, 128, 8192
    dims = pa.make_dims(nb, bs, 28, hkv, d)
    kc = torch.empty(nb, bs, hkv, d, dtype=torch.bfloat16, device=device).normal_()
    vc = torch.empty_like(kc).normal_()
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    trip = torch.stack([perm[:n], perm[n:], torch.full((n,), bs, dtype=torch.int32)], 1).contiguous().to(device)
    for _ in range(warmup):
        pa.pa_copy_blocks(dims, kc, vc, trip, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in evs:
        a.record(stream)
        pa.pa_copy_blocks(dims, kc, vc, trip, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    work = 2.0 * n * bs * hkv * d * 2 * 2  # K and V rows, read and written
    gbs = work / (ms * 1e-3) / 1e9
    return {"kernel": "pa_copy_blocks (copy_blocks_kernel)", "bound": "hbm", "achieved": round(gbs, 1),
            "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "peak_source": f"{peak_src} hbm_gbs",
            "traffic": NCU_TRAFFIC_COPY_BLOCKS, "work_per_launch": work, "ms_per_launch": round(ms, 5),
            "workload": "8192 full-block copies (block 16, 4 KV heads, D 128), 256 MB read + 256 MB written"}


def read_stream_gbs(pool, stream, int8, step, iters=10, warmup=3):
    """Read-only bandwidth over the decode cache's own buffers (pa_stream_read), CUDA events."""
    from paged_kv_cache_kvcache_gb300 import pagedattn as pa
    bufs = list(step.c8_d) if int8 else [pool.k_cache, pool.v_cache]
    bufs = [b for b in bufs if b.numel() * b.element_size() % 16 == 0]
    sink = torch.zeros(1, dtype=torch.int32, device=pool.k_cache.device)
    nbytes = sum(b.numel() * b.element_size() for b in bufs)
    for _ in range(warmup):
        for b in bufs:
            pa.pa_stream_read(b, sink, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        for b in bufs:
            pa.pa_stream_read(b, sink, stream=stream)
    e1.record(stream)
    e1.synchronize()
    return round(nbytes * iters / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)


def oracle_prefill_sample(wp, row_stride, threads=0):
    """Oracle on every row_stride-th query row of the prefill batch; returns (seconds, flops)."""
    import oracle
    b = wp.batches[0]
    sel = np.zeros(b.num_tokens, dtype=bool)
    sel[::row_stride] = True
    kb = wp.pool.k_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    vb = wp.pool.v_cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    t0 = time.perf_counter()
    _, pairs = oracle.run_batch(kb, vb, b, wp.pool.block_size, row_select=sel, num_threads=threads)
    dt = time.perf_counter() - t0
    return dt, 4.0 * b.q.shape[2] * pairs


def oracle_decode_sample(wd, nseq, threads=0):
    """Oracle decode on the first nseq sequences; returns (seconds, KV bytes read by the method)."""
    import oracle
    from paged_kv_cache_kvcache_gb300 import workloads
    b = wd.batches[0]
    seqs = list(range(nseq))
    used = np.unique(np.concatenate([b.block_lists[i] for i in seqs]))
    remap = {int(p): i for i, p in enumerate(used)}
    idx = torch.from_numpy(used.astype(np.int64)).to(wd.pool.k_cache.device)
    kb = wd.pool.k_cache.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    vb = wd.pool.v_cache.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    sub = workloads.Batch("decode", b.seq_lens[seqs], b.query_lens[seqs],
                          [np.array([remap[int(p)] for p in b.block_lists[i]], np.int32) for i in seqs],
                          b.q[seqs].cpu(), b.k[seqs].cpu(), b.v[seqs].cpu(), b.num_heads, b.scale)
    t0 = time.perf_counter()
    oracle.run_batch(kb, vb, sub, wd.pool.block_size, num_threads=threads)
    dt = time.perf_counter() - t0
    kv = float(np.sum(sub.seq_lens.astype(np.int64))) * wd.pool.num_kv_heads * wd.pool.head_dim * 4
    return dt, kv


# ---------------------------------------------------------------- main


def main():
    args = parse()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"
    assert args.decode_path != "mixed" or (args.kv == "bf16" and args.phase == "both"), \
        "--decode-path mixed runs the bf16 cache, both phases"
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks, peak_src = load_peaks()
    wp, wd, wl_desc = make_workload(args.workload, f"cuda:{local}", args.decode_seqs)
    stream = torch.cuda.Stream()
    clocks = Clocks(local, enabled=not args.no_clocks)
    with torch.cuda.stream(stream):
        step = Step(wp, wd, stream, kv=args.kv, fused=args.decode_path == "fused",
                    mixed=args.decode_path == "mixed", prefill_fused=args.prefill_path == "fused")
        names = ["p0", "pk0", "pk1", "p1", "dk0", "dk1", "d1"]
        for _ in range(args.warmup):
            step.run(phase=args.phase)
        stream.synchronize()
        evs = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(args.steps)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        t_start.record(stream)
        for i in range(args.steps):
            step.run(evs[i], phase=args.phase)
        t_end.record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        # every kernel hand-off waits with a time limit; a wait that ran out leaves its
        # outputs undefined and is recorded in the device error word: such a run is invalid
        derr = step.pa.pa_read_device_error(stream)
        if derr:
            raise RuntimeError(f"device error word {derr:#x} after the timed steps: outputs undefined")
        if world > 1:
            torch.distributed.barrier()
        clk = clocks.stop(w0, w1)
        total_ms = max_over_ranks(t_start.elapsed_time(t_end))
        ph = lambda a, b: [e[a].elapsed_time(e[b]) for e in evs]
        t_prefill_phase = statistics.mean(ph("p0", "p1"))
        t_prefill_kernel = statistics.mean(ph("pk0", "pk1"))
        t_decode_phase = statistics.mean(ph("p1", "d1"))
        t_decode_kernel = statistics.mean(ph("dk0", "dk1"))

        # e2e: the same step through the public API with host (pinned) inputs/outputs
        # mixed: the same rows as separate prefill and decode launches, timed the same way
        separate = None
        if args.decode_path == "mixed":
            ref_step = Step(wp, wd, stream)
            for _ in range(args.warmup):
                ref_step.run()
            evs3 = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(args.steps)]
            for i in range(args.steps):
                ref_step.run(evs3[i])
            torch.cuda.synchronize()
            ph3 = lambda a, b: statistics.mean([e[a].elapsed_time(e[b]) for e in evs3])
            separate = {"prefill_kernel_ms": round(ph3("pk0", "pk1"), 5), "decode_kernels_ms": round(ph3("dk0", "dk1"), 5),
                        "step_ms": round(ph3("p0", "d1"), 5)}

        e2e = None
        if not args.no_e2e and args.phase == "both" and args.decode_path != "mixed":
            e2e_p, h2d_p, d2h_p = pipelined_e2e(step, "p", args.steps, args.warmup)
            e2e_d, h2d_d, d2h_d = pipelined_e2e(step, "d", args.steps, args.warmup)
            meta_bytes = int(step.plans_p[0].meta.total_bytes + step.plans_d[0].meta.total_bytes)
            e2e = {"value": round(prefill_flops(step.bp) / (e2e_p * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d_p + h2d_d + meta_bytes, "d2h_bytes_per_step": d2h_p + d2h_d,
                   "decode": {"value": round(decode_bytes(step.bd, wd.pool, args.kv) / (e2e_d * 1e-3) / 1e9 * world,
                                             1),
                              "unit": "GB/s"},
                   "ms_per_step": round(e2e_p + e2e_d, 4),
                   "pipelining": "per phase: step i+1's inputs copied in and step i-1's output copied out "
                                 "(pinned host memory, one copy stream each way) while step i computes"}

    flops = prefill_flops(step.bp)
    dbytes = decode_bytes(step.bd, wd.pool, args.kv)
    eps = 1e-9  # a phase left out with --phase times as ~0
    value = flops / (max(t_prefill_phase, eps) * 1e-3) / 1e12 * world
    decode_gbs = dbytes / (max(t_decode_phase, eps) * 1e-3) / 1e9 * world
    if args.decode_path == "mixed":  # one phase holds both: rates over that phase
        flops = prefill_flops(step.bm)
        value = flops / (t_prefill_phase * 1e-3) / 1e12 * world
        decode_gbs = dbytes / (t_prefill_phase * 1e-3) / 1e9 * world
    pk_tflops = flops / (max(t_prefill_kernel, eps) * 1e-3) / 1e12
    dk_gbs = dbytes / (max(t_decode_kernel, eps) * 1e-3) / 1e9
    t_decode_phase = max(t_decode_phase, eps)
    t_prefill_phase = max(t_prefill_phase, eps)
    bf16_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    int8 = args.kv == "int8"
    traffic = {} if args.decode_path in ("fused", "mixed") else \
        (NCU_TRAFFIC_INT8 if int8 else NCU_TRAFFIC).get(args.workload, {})
    if step.prefill_fused:
        traffic = {"prefill": (NCU_TRAFFIC_INT8_FUSED_PREFILL if int8 else NCU_TRAFFIC_FUSED_PREFILL).get(args.workload),
                   "decode": traffic.get("decode")}
    if int8:
        pk_name = ("pa_prefill_varlen_int8_fused (int8_gather_kernel<128,true>: quantising store of the new rows "
                   "+ bf16 dequantisation into the scratch cache; then prefill_kernel<128,false>)" if step.prefill_fused else
                   "pa_prefill_varlen_int8 (int8_gather_kernel<128,false>: bf16 dequantisation into the scratch "
                   "cache; then prefill_kernel<128,false>)")
    else:
        pk_name = ("pa_prefill_varlen_fused (prefill_kernel<128,false>, store of the new K/V fused)"
                   if step.prefill_fused else "pa_prefill_varlen (prefill_kernel<128,false>)")
    roof_p = {"kernel": pk_name,
              "bound": "tensor", "achieved": round(pk_tflops, 2),
              "peak": bf16_peak, "unit": "TFLOP/s", "frac": round(pk_tflops / bf16_peak, 4),
              "peak_source": f"{peak_src} bf16_tflops (burst; f16 has the same nominal rate)",
              "traffic": traffic.get("prefill"),
              "work_per_launch": flops, "ms_per_launch": round(t_prefill_kernel, 5)}
    dk_name = {"bf16": "pa_decode (decode_split_kernel<128,1,false> + decode_combine_kernel<128>)",
               "int8": "pa_decode_int8 (decode_int8_kernel<128,1> + decode_combine_kernel<128>)"}[args.kv]
    if args.decode_path == "fused":
        dk_name = ("pa_decode_int8_fused (decode_int8_kernel<128,1,true> + decode_combine_kernel<128>)" if int8 else
                   "pa_decode_fused (decode_split_kernel<128,1,true> + decode_combine_kernel<128>)")
    roof_d = {"kernel": dk_name, "bound": "hbm",
              "achieved": round(dk_gbs, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(dk_gbs / hbm_peak, 4),
              "peak_source": f"{peak_src} hbm_gbs",
              "traffic": traffic.get("decode") if args.decode_seqs == 64 else None,
              "work_per_launch": dbytes, "ms_per_launch": round(t_decode_kernel, 5)}
    # The decode reads its cache and writes little: besides the copy peak (read + write,
    # the headline denominator), report it against a read-only stream over the same
    # cache buffers measured now on this GPU, and against the nominal HBM3e rate.
    if args.decode_path != "mixed" and args.phase in ("both", "decode"):
        with torch.cuda.stream(stream):
            rs = read_stream_gbs(wd.pool, stream, args.kv == "int8", step)
        roof_d["denominators"] = {
            "headline": "frac: against the measured copy peak (MEASURED_PEAKS hbm_gbs, read + write)",
            "read_stream_gbs": rs, "frac_of_read_stream": round(dk_gbs / rs, 4),
            "read_stream_how": "pa_stream_read over the decode cache buffers (16-byte streaming loads, "
                               "the same bytes the decode reads), CUDA events, this run",
            "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": round(dk_gbs / NOMINAL_HBM_GBS, 4)}
    dominant = roof_p if t_prefill_kernel >= t_decode_kernel else roof_d
    rooflines = [roof_p, roof_d]
    if args.phase == "both" and args.decode_path == "store+decode" and args.kv == "bf16":
        with torch.cuda.stream(stream):
            rooflines.append(copy_blocks_roofline(f"cuda:{local}", stream, hbm_peak, peak_src))
    mixed = None
    if args.decode_path == "mixed":
        # One launch holds compute-bound prefill rows and bandwidth-bound decode rows: its
        # lower bound is the prefill rows' FLOPs at the tensor peak plus the decode rows'
        # K/V bytes at the copy peak.  The roofline entry counts the decode bytes (the larger part).
        pf = prefill_flops(step.bp)
        t_low = (pf / (bf16_peak * 1e12) + dbytes / (hbm_peak * 1e9)) * 1e3
        gbs = dbytes / (t_prefill_kernel * 1e-3) / 1e9
        roof_p = {"kernel": "pa_prefill_varlen (prefill_kernel<128,false>), prefill + decode rows", "bound": "hbm",
                  "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                  "peak_source": f"{peak_src} hbm_gbs", "traffic": None, "work_per_launch": dbytes,
                  "ms_per_launch": round(t_prefill_kernel, 5)}
        dominant, rooflines = roof_p, [roof_p]
        mixed = {"kernel_ms": round(t_prefill_kernel, 5), "phase_ms": round(t_prefill_phase, 5),
                 "rows": {"prefill_tokens": int(step.bp.num_tokens), "decode_rows": int(step.bd.num_seqs)},
                 "lower_bound_ms": round(t_low, 5), "frac_of_lower_bound": round(t_low / t_prefill_kernel, 4),
                 "separate": separate}

    cpu = None
    # the CPU leg times the bf16 oracle on the default path only
    if (rank == 0 and not args.no_cpu_baseline and world == 1 and args.phase == "both" and args.kv == "bf16"
            and args.decode_path == "store+decode"):
        import oracle
        dt_p, fl = oracle_prefill_sample(wp, row_stride=1)
        dt_d, kvb = oracle_decode_sample(wd, nseq=16)
        cpu = {"value": round(fl / dt_p / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
               "omp_threads": oracle.max_threads(), "cpu_count": os.cpu_count(),
               "kind": "oracle",
               "sample": f"prefill: the whole 4x4096 batch ({fl / 1e9:.1f} GFLOP, {dt_p:.1f} s); "
                         f"decode: 16 of 64 sequences ({kvb / 1e9:.2f} GB K/V, {dt_d:.1f} s)",
               "decode": {"value": round(kvb / dt_d / 1e9, 3), "unit": "GB/s"}}
        # one host thread, on smaller samples (every 64th prefill row, 2 decode sequences)
        dt_p1, fl1 = oracle_prefill_sample(wp, row_stride=64, threads=1)
        dt_d1, kvb1 = oracle_decode_sample(wd, nseq=2, threads=1)
        cpu["single_thread"] = {"value": round(fl1 / dt_p1 / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                                "sample": f"prefill: every 64th query row ({fl1 / 1e9:.1f} GFLOP, {dt_p1:.1f} s); "
                                          f"decode: 2 sequences ({kvb1 / 1e9:.2f} GB K/V, {dt_d1:.1f} s)",
                                "decode": {"value": round(kvb1 / dt_d1 / 1e9, 3), "unit": "GB/s"}}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 KV (prefill: bf16 dequantised; decode: f16 MMA)" if int8 else "bf16", "data": "synthetic",
        "config": {"workload": wl_desc, "l2": "inputs larger than L2: the decode phase streams "
                   f"{dbytes / 1e9:.2f} GB per step", "prefill_gflop": round(flops / 1e9, 2),
                   "decode_kv_gb": round(dbytes / 1e9, 3), "parallelism": f"replicas x{world}", "kv": args.kv,
                   "decode_path": args.decode_path, "prefill_path": "fused" if step.prefill_fused else "store+prefill"},
        "decode": {"value": round(decode_gbs, 1), "unit": "GB/s", "frac_of_hbm": round(decode_gbs / hbm_peak, 4),
                   "seqs_per_s": round(step.bd.num_seqs / (t_decode_phase * 1e-3) * world, 1)},
        "prefill": {"tokens_per_s": round(step.bp.num_tokens / (t_prefill_phase * 1e-3) * world, 1),
                    "frac_of_bf16": round(value / world / bf16_peak, 4)},
        "phase_ms": {"prefill_phase": round(t_prefill_phase, 5), "prefill_kernel": round(t_prefill_kernel, 5),
                     "decode_phase": round(t_decode_phase, 5), "decode_kernels": round(t_decode_kernel, 5)},
        "roofline": dominant, "rooflines": rooflines,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clk, "peaks": peak_src, "device_error": 0,
    }
    if mixed is not None:
        line["mixed"] = mixed
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def reference_arm(args, rank, world):
    """The CPU oracle, as it stands, timed on the host cores on bounded samples of the same workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    device = "cuda" if torch.cuda.is_available() else "cpu"
    wp, wd, wl_desc = make_workload(args.workload, device, args.decode_seqs)
    # size each step's sample so that the whole --warmup + --steps run takes about 90 s
    budget = max(0.05, 90.0 / (args.warmup + args.steps))
    t_cal, _ = oracle_prefill_sample(wp, row_stride=1024)
    stride = int(min(16384, max(16, 1024 * t_cal / (0.7 * budget))))
    t_dec, _ = oracle_decode_sample(wd, nseq=1)
    dec_every = max(1, int(round(t_dec / (0.3 * budget))))
    sp, sd = [], []
    for i in range(args.warmup + args.steps):
        dt_p, fl = oracle_prefill_sample(wp, row_stride=stride)
        dt_d, kvb = oracle_decode_sample(wd, nseq=1) if i % dec_every == 0 else (0.0, 0.0)
        if i >= args.warmup:
            sp.append((dt_p, fl))
            if kvb:
                sd.append((dt_d, kvb))
    if not sd:
        sd.append(oracle_decode_sample(wd, nseq=1))
    tp = sum(x[0] for x in sp)
    value = sum(x[1] for x in sp) / tp / 1e12
    td = sum(x[0] for x in sd)
    dec = sum(x[1] for x in sd) / td / 1e9
    cores = oracle.max_threads()
    sample = (f"per step: every {stride}th query row of the 4x4096 prefill batch; 1 of the 64 decode sequences "
              f"every {dec_every} step(s) ({wl_desc})")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round((tp + td) / len(sp) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl_desc, "parallelism": "cpu oracle"},
            "decode": {"value": round(dec, 3), "unit": "GB/s"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "omp_threads": cores,
                             "cpu_count": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
