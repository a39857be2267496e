"""Invariants the PagedAttention pages fix, checked on the GPU, plus the
degenerate and faulting inputs.

The block table is an indirection only (Qualiteg, "About PagedAttention for
LLM serving", the section on logical and physical blocks), so any physical
placement of the same tokens must
give bitwise the same output: the kernel's arithmetic order depends only on
logical positions.  Sequences that share prefix blocks (the prefix-sharing
use discussed on the Hacker News page) must give bitwise the result of
private copies.  Faults are made on the host (bad table entries, bad
lengths): they must be reported in the error word, never trap.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write, run_decode

pytestmark = pytest.mark.gpu


def _replace(w, placement_seed):
    """Same logical tokens, other physical blocks (pool twice as large)."""
    NB2 = w.num_blocks * 2
    perm = np.random.default_rng(placement_seed).permutation(NB2)[: w.num_blocks]
    kp = torch.full((NB2,) + tuple(w.k_pool.shape[1:]), float("nan"), dtype=w.k_pool.dtype)
    vp = torch.full_like(kp, float("nan"))
    kp[torch.from_numpy(perm)] = w.k_pool
    vp[torch.from_numpy(perm)] = w.v_pool
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    sm = np.where(w.slot_mapping >= 0,
                  perm[w.slot_mapping // w.block_size] * w.block_size + w.slot_mapping % w.block_size,
                  -1)
    import dataclasses
    return dataclasses.replace(w, k_pool=kp, v_pool=vp, block_tables=bt, slot_mapping=sm,
                               num_blocks=NB2)


@pytest.mark.parametrize("dtype,H,Hkv,BS", [("bf16", 32, 8, 16), ("bf16", 16, 16, 16),
                                            ("f32", 8, 2, 16), ("f16", 32, 8, 16),
                                            ("bf16", 32, 8, 64)])
@pytest.mark.parametrize("partition", [-1, 256])
def test_placement_invariance_bitwise(dtype, H, Hkv, BS, partition):
    w = workload.build("perm", dtype=dtype, context_lens=[3, 200, 1000, 47, 512], num_heads=H,
                       num_kv_heads=Hkv, head_dim=128, block_size=BS, data_seed=11, meta_seed=12)
    base = run_decode(w, partition_tokens=partition).out.cpu()
    for seed in (1, 2):
        other = run_decode(_replace(w, seed), partition_tokens=partition).out.cpu()
        assert torch.equal(base.view(torch.int32), other.view(torch.int32))


@pytest.mark.parametrize("partition", [-1, 0, 1024])
def test_shared_prefix_equals_private_copies_bitwise(partition):
    ctx = [2048 + 37, 2048 + 100, 2048 + 1, 2048 + 400]
    w = workload.build("share", dtype="bf16", context_lens=ctx, num_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=16, data_seed=21, meta_seed=22, group_size=2,
                       prefix_len=2048)
    shared = run_decode(w, partition_tokens=partition)
    ref, _, _ = oracle_after_write(w)
    assert_close(shared.out, ref, "bf16", "shared prefix")
    # private copies of the prefix blocks for the second member of each group
    kp, vp, bt = [w.k_pool], [w.v_pool], w.block_tables.copy()
    nb = w.num_blocks
    for s in (1, 3):
        for b in range(2048 // 16):
            kp.append(w.k_pool[bt[s, b]][None])
            vp.append(w.v_pool[bt[s, b]][None])
            bt[s, b] = nb
            nb += 1
    import dataclasses
    wp = dataclasses.replace(w, k_pool=torch.cat(kp), v_pool=torch.cat(vp), block_tables=bt,
                             num_blocks=nb)
    private = run_decode(wp, partition_tokens=partition)
    assert torch.equal(shared.out.cpu().view(torch.int32), private.out.cpu().view(torch.int32))


def test_split_and_single_pass_agree():
    w = workload.build("split", dtype="bf16", context_lens=[4000, 1500, 7000, 33], num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=31, meta_seed=32)
    a = run_decode(w, partition_tokens=-1).out.double()
    for pt in (256, 512, 4096):
        b = run_decode(w, partition_tokens=pt).out.double()
        assert float((a - b).abs().max()) <= 2e-3


def test_fma_and_mma_paths_agree():
    w = workload.build("paths", dtype="bf16", context_lens=[800, 15, 2500], num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=41, meta_seed=42)
    ref, _, _ = oracle_after_write(w)
    for path in (pagedkv.PATH_FMA, pagedkv.PATH_MMA):
        assert_close(run_decode(w, path=path).out, ref, "bf16", f"path {path}")


def test_nan_in_unused_slots_is_ignored():
    for dtype, H, Hkv in (("bf16", 32, 8), ("bf16", 8, 8), ("f32", 4, 2), ("f32", 16, 2)):
        w = workload.build("nan", dtype=dtype, context_lens=[17, 5, 250, 33], num_heads=H,
                           num_kv_heads=Hkv, head_dim=128, block_size=16, data_seed=51,
                           meta_seed=52, pool_blocks=40, tail_fill=float("nan"))
        ref, _, _ = oracle_after_write(w)
        for pt in (-1, 64):
            dw = run_decode(w, partition_tokens=pt)
            assert_close(dw.out, ref, dtype, f"nan tails {dtype} G{H // Hkv} pt {pt}")


def test_empty_context_gives_zeros():
    w = workload.build("empty", dtype="bf16", context_lens=[0, 40, 0, 600], num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=61, meta_seed=62)
    ref, _, _ = oracle_after_write(w)
    for pt in (-1, 0, 128):
        dw = run_decode(w, partition_tokens=pt)
        assert torch.all(dw.out[0] == 0) and torch.all(dw.out[2] == 0)
        assert_close(dw.out, ref, "bf16", "empty contexts")


def test_context_at_table_capacity():
    # every sequence fills its whole block table (max_blocks_per_seq * BS tokens)
    w = workload.build("full", dtype="bf16", context_lens=[1024, 1024], num_heads=16,
                       num_kv_heads=4, head_dim=128, block_size=32, data_seed=71, meta_seed=72,
                       max_blocks_per_seq=32)
    ref, _, _ = oracle_after_write(w)
    for pt in (-1, 0, 256):
        dw = run_decode(w, partition_tokens=pt)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, "bf16", "full table")


def test_bad_block_id_sets_fault_and_spares_other_sequences():
    w = workload.build("badblk", dtype="bf16", context_lens=[100, 300, 64], num_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=81, meta_seed=82)
    ref, _, _ = oracle_after_write(w)
    dw = pagedkv.DeviceWorkload(w)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    bt = dw.block_tables.clone()
    bt[1, 3] = w.num_blocks + 5  # outside the pool
    for pt in (-1, 0, 64):
        pagedkv.paged_attention_decode(dw.pool, dw.out, dw.q, bt, dw.context_lens, 300, w.scale,
                                       partition_tokens=pt, workspace=pagedkv.alloc_workspace(
                                           3, 32, 128, 300, pt))
        assert pagedkv.get_device_error(dw.pool) == pagedkv.FAULT_BLOCK_ID
        out = dw.out.cpu()
        assert torch.isfinite(out).all()
        for s in (0, 2):
            assert_close(out[s], ref[s], "bf16", f"unaffected sequence {s}")


def test_context_beyond_bound_sets_fault_and_clamps():
    w = workload.build("badctx", dtype="bf16", context_lens=[100, 300], num_heads=8,
                       num_kv_heads=8, head_dim=128, block_size=16, data_seed=91, meta_seed=92)
    dw = pagedkv.DeviceWorkload(w)
    pagedkv.paged_attention_decode(dw.pool, dw.out, dw.q, dw.block_tables, dw.context_lens, 200,
                                   w.scale, partition_tokens=-1)
    assert pagedkv.get_device_error(dw.pool) == pagedkv.FAULT_CONTEXT
    cl = dw.context_lens.clone()
    cl[0] = -5
    pagedkv.paged_attention_decode(dw.pool, dw.out, dw.q, dw.block_tables, cl, 300, w.scale,
                                   partition_tokens=-1)
    assert pagedkv.get_device_error(dw.pool) == pagedkv.FAULT_CONTEXT
    assert torch.all(dw.out[0] == 0)


def test_workspace_too_small_is_rejected():
    w = workload.build("ws", dtype="bf16", context_lens=[2000], num_heads=8, num_kv_heads=8,
                       head_dim=128, block_size=16, data_seed=1, meta_seed=2)
    dw = pagedkv.DeviceWorkload(w)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pagedkv.PagedKVError) as e:
        pagedkv.paged_attention_decode(dw.pool, dw.out, dw.q, dw.block_tables, dw.context_lens,
                                       2000, w.scale, partition_tokens=512, workspace=small)
    assert e.value.status == pagedkv.ERR_WORKSPACE
