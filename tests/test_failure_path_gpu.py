"""The library's failure path, exercised without a fault: a bounded mbarrier wait
that nothing completes gives up after its time limit, the kernel records that in
the device error word and returns, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvcache_gb300 import pagedattn as pa
from paged_kv_cache_kvcache_gb300 import workloads
from tests.harness import assert_close, bits, run_gpu_batch

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 1 << 4


def test_bounded_wait_completed_barrier_reports_nothing():
    assert pa.pa_read_device_error() == 0
    pa.pa_selftest_bounded_wait(20000, arrive_first=True)
    assert pa.pa_read_device_error() == 0


def test_bounded_wait_times_out_reports_and_the_context_stays_usable():
    assert pa.pa_read_device_error() == 0
    t0 = time.perf_counter()
    pa.pa_selftest_bounded_wait(20000)  # 20 ms on a barrier nothing completes
    code = pa.pa_read_device_error()
    dt = time.perf_counter() - t0
    assert code == SELFTEST_BIT
    assert 0.015 < dt < 5.0
    assert pa.pa_read_device_error() == 0  # read and cleared
    # the same process then runs real work correctly
    w = workloads.random_case(141, num_seqs=4, hq=8, hkv=2, d=128, bs=16, max_len=300, device="cuda")
    batch = w.batches[0]
    kc, vc = w.pool.k_cache.clone(), w.pool.v_cache.clone()
    out, _ = run_gpu_batch(w, batch, kc, vc)
    ref, _ = oracle.run_batch(bits(w.pool.k_cache), bits(w.pool.v_cache), batch, w.pool.block_size)
    torch.cuda.synchronize()
    assert pa.pa_read_device_error() == 0
    assert_close(out, ref, what="after a timed-out wait")
