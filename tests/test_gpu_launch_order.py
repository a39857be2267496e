"""Inputs written by the kernel right before a decode are what the decode
reads.

The decode and combine kernels are launched as programmatic dependents of
the kernel before them in the stream and wait (griddepcontrol.wait) before
reading any input; these tests change the query, the context lengths and the
block tables with ordinary device kernels immediately before each decode,
with no synchronisation in between, and check the result against the
oracle on the changed inputs.
"""
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


def _w(**kw):
    return workload.build("order", dtype="bf16", context_lens=[300, 1200, 47, 2000, 900],
                          num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          data_seed=71, meta_seed=72, **kw)


@pytest.mark.parametrize("partition", [-1, 256])
def test_decode_sees_query_written_just_before(partition):
    w = _w()
    dw = pagedkv.DeviceWorkload(w, partition_tokens=partition)
    dw.step()
    for scale in (2.0, -0.5, 3.0):
        dw.q.mul_(scale)  # a device kernel right before the decode
        dw.decode()
        torch.cuda.synchronize()
        w.q = dw.q.cpu()  # the oracle sees the same (rounded) query
        ref, _, _ = oracle_after_write(w)
        assert_close(dw.out, ref, "bf16", f"query x{scale}")


def test_decode_sees_context_lengths_and_tables_written_just_before():
    w = _w()
    dw = pagedkv.DeviceWorkload(w, partition_tokens=256)
    dw.step()
    # shorten every context by a few tokens and swap two sequences' tables on the device
    dw.context_lens.sub_(torch.tensor([5, 17, 0, 300, 1], dtype=torch.int32, device="cuda"))
    dw.block_tables[[0, 2]] = dw.block_tables[[2, 0]]
    dw.context_lens[[0, 2]] = dw.context_lens[[2, 0]].clone()
    dw.decode()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    import dataclasses
    w2 = dataclasses.replace(w, context_lens=dw.context_lens.cpu().numpy(),
                             block_tables=dw.block_tables.cpu().numpy())
    # the pool already holds the step's new tokens; compare without writing again
    import oracle
    ref = oracle.paged_decode(w2.q, dw.k_pool.cpu(), dw.v_pool.cpu(), w2.block_tables,
                              w2.context_lens, w2.scale)
    assert_close(dw.out, ref, "bf16", "changed lengths and tables")


def test_shared_prefix_decode_sees_query_written_just_before():
    ctx = [256 + s for s in (3, 40, 100, 7, 64, 1)]
    w = workload.build("order_sp", dtype="bf16", context_lens=ctx, num_heads=16, num_kv_heads=4,
                       head_dim=128, block_size=16, data_seed=73, meta_seed=74,
                       groups=[(4, 256), (2, 256)])
    dw = pagedkv.DeviceWorkload(w)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    dw.shared_prefix_setup()
    dw.decode_shared_prefix()
    dw.q.mul_(-2.0)
    dw.decode_shared_prefix()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    w.q = dw.q.cpu()
    ref, _, _ = oracle_after_write(w)
    assert_close(dw.out, ref, "bf16", "shared prefix, query x-2")
