"""The kernels' watchdog, exercised without a GPU fault.

Every shared-memory pipeline wait of the decode kernels is bounded: past its
limit the kernel records PKV_FAULT_TIMEOUT and stops, so a copy that never
lands cannot hang the GPU.  pkv_check_bounded_wait runs that same wait on a
barrier nothing arrives at (a flag that nothing sets), with a short bound;
the fault bit must come back, and the context must still run a decode that
matches the oracle.
"""
import time

import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    w = workload.build("watchdog", dtype="bf16", context_lens=[5, 300, 1200], num_heads=16,
                       num_kv_heads=4, head_dim=128, block_size=16, data_seed=800, meta_seed=801)
    dw = pagedkv.DeviceWorkload(w, partition_tokens=256)
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    limit_ns = 20_000_000
    t0 = time.perf_counter()
    pagedkv.check_bounded_wait(dw.pool, limit_ns)
    bits = pagedkv.get_device_error(dw.pool)  # synchronises
    elapsed = time.perf_counter() - t0
    assert bits == pagedkv.FAULT_TIMEOUT
    assert limit_ns * 1e-9 <= elapsed < 1.5, elapsed
    # the error word was cleared by the read, and the context still works
    dw.step()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    ref, _, _ = oracle_after_write(w)
    assert_close(dw.out, ref, "bf16", "decode after the watchdog check")
