"""The allocation-free decode entry point, for callers that cannot allocate
device memory (an engine that hands all device memory to its KV pool and a
caching allocator at start-up, a plain-C host without a device allocator, a
latency-critical loop where cudaMalloc would synchronise the device).

Called through the C ABI; its output must match the workspace-taking entry
point's within the parity tolerance, on two calls in a row (the second call
finds the first call's partials still in the shared scratch array).  This
file is collected last so that a stop-at-first-failure run has already run
every other test.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write


def _call_static(lib, dw, out, partition):
    w = dw.w
    return lib.pkv_paged_attention_decode_static(
        ctypes.byref(dw.pool.desc), out.data_ptr(), pagedkv.F32, dw.q.data_ptr(), w.num_seqs,
        w.num_heads, w.num_kv_heads, dw.block_tables.data_ptr(), w.max_blocks_per_seq,
        dw.context_lens.data_ptr(), dw.max_context_len, w.scale, partition, pagedkv.PATH_AUTO,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    lib = pagedkv.load()
    cases = [
        workload.build("noalloc_gqa", dtype="bf16", context_lens=[3000, 17, 1200, 5000, 1],
                       num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, data_seed=5,
                       meta_seed=6),
        workload.build("noalloc_mha", dtype="bf16", context_lens=[700, 2048, 129], num_heads=16,
                       num_kv_heads=16, head_dim=128, block_size=16, data_seed=7, meta_seed=8),
    ]
    for w in cases:
        ref, _, _ = oracle_after_write(w)
        for partition in (0, 256):
            dw = pagedkv.DeviceWorkload(w, partition_tokens=partition)
            pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
            dw.decode()  # the existing entry point, caller-owned workspace
            torch.cuda.synchronize()
            expect = dw.out.clone()
            assert_close(expect, ref, "bf16", f"{w.name} workspace entry point")
            for call in range(2):
                got = torch.full_like(dw.out, float("nan"))
                assert _call_static(lib, dw, got, partition) == pagedkv.OK
                torch.cuda.synchronize()
                assert pagedkv.get_device_error(dw.pool) == 0
                assert_close(got, expect.double().cpu().numpy(), "bf16",
                             f"{w.name} partition {partition} call {call}")
                assert_close(got, ref, "bf16", f"{w.name} vs oracle, call {call}")


@pytest.mark.gpu
def test_static_scratch_rejects_partials_beyond_its_size():
    lib = pagedkv.load()
    w = workload.build("noalloc_big", dtype="bf16", context_lens=[64], num_heads=64,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=9, meta_seed=10)
    dw = pagedkv.DeviceWorkload(w)
    # 8 x 64 heads x 1024 partitions of 16 tokens x 129 floats > 64 MiB
    need = pagedkv.decode_workspace_bytes(8, 64, 128, 16384, 16)
    assert need > pagedkv.STATIC_SCRATCH_BYTES
    q = torch.zeros(8, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(8, 64, 128, dtype=torch.float32, device="cuda")
    bt = torch.zeros(8, 1024, dtype=torch.int32, device="cuda")
    cl = torch.ones(8, dtype=torch.int32, device="cuda")
    st = lib.pkv_paged_attention_decode_static(
        ctypes.byref(dw.pool.desc), out.data_ptr(), pagedkv.F32, q.data_ptr(), 8, 64, 8,
        bt.data_ptr(), 1024, cl.data_ptr(), 16384, w.scale, 16, pagedkv.PATH_AUTO,
        torch.cuda.current_stream().cuda_stream)
    assert st == pagedkv.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched


@pytest.mark.gpu
def test_static_scratch_long_context_automatic_partition():
    """The full long-context batch (8 sequences of 32k-128k tokens, 64/8
    heads) with the automatic partition: the decode takes 1024- or
    2048-token partitions whose partials fit in the fixed array, although
    the workspace bound for 512-token partitions does not."""
    lib = pagedkv.load()
    w = workload.make("long_ctx", partition_tokens=0)
    assert pagedkv.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim,
                                          w.max_context_len, 0) > pagedkv.STATIC_SCRATCH_BYTES
    ref, _, _ = oracle_after_write(w)
    dw = pagedkv.DeviceWorkload(w, partition_tokens=0)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    dw.decode()
    torch.cuda.synchronize()
    expect = dw.out.clone()
    assert_close(expect, ref, "bf16", "long_ctx workspace entry point")
    for call in range(2):
        got = torch.full_like(dw.out, float("nan"))
        assert _call_static(lib, dw, got, 0) == pagedkv.OK
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        assert torch.equal(got, expect), f"long_ctx call {call}: differs from the workspace call"
        assert_close(got, ref, "bf16", f"long_ctx vs oracle, call {call}")
