"""Element-by-element parity of the CUDA path with the float64 oracle.

Cache writes are compared byte for byte over the whole pool; attention
outputs within 1e-5 (fp32 inputs) or 2e-3 (bf16 inputs, fp32 accumulation),
on sizes that span several tiles, partitions and a ragged last block.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write, run_decode

pytestmark = pytest.mark.gpu

RAGGED = [1, 15, 16, 17, 100, 333, 700]


def _w(dtype, D, BS, H, Hkv, ctx=RAGGED, seed=0, **kw):
    return workload.build(f"parity_{dtype}_d{D}_bs{BS}_h{H}_{Hkv}", dtype=dtype, context_lens=ctx,
                          num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=BS,
                          data_seed=1000 + seed, meta_seed=2000 + seed, **kw)


# ------------------------------------------------------------ cache write --

@pytest.mark.parametrize("dtype,D,BS", [("f32", 64, 16), ("bf16", 128, 16), ("bf16", 64, 32),
                                        ("f32", 128, 32), ("f16", 128, 16), ("f16", 64, 64)])
def test_reshape_and_cache_bit_exact(dtype, D, BS):
    w = _w(dtype, D, BS, 8, 4, ctx=[1, 16, 17, 40, 64, 65], pool_blocks=30)
    sm = w.slot_mapping.copy()
    sm[1] = -1                          # padding token: skipped
    dw = pagedkv.DeviceWorkload(w)
    dw.slot_mapping.copy_(torch.from_numpy(sm))
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, sm) == 0
    view = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(dw.k_pool.cpu().view(view), kp.view(view))
    assert torch.equal(dw.v_pool.cpu().view(view), vp.view(view))


def test_reshape_and_cache_slot_past_pool_faults_and_skips():
    w = _w("bf16", 128, 16, 8, 2, ctx=[5, 20, 33])
    sm = w.slot_mapping.copy()
    sm[2] = w.num_blocks * w.block_size  # one past the last slot
    dw = pagedkv.DeviceWorkload(w)
    dw.slot_mapping.copy_(torch.from_numpy(sm))
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    assert pagedkv.get_device_error(dw.pool) == pagedkv.FAULT_SLOT
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, sm) == 1
    assert torch.equal(dw.k_pool.cpu().view(torch.int16), kp.view(torch.int16))
    assert torch.equal(dw.v_pool.cpu().view(torch.int16), vp.view(torch.int16))


# ---------------------------------------------------------------- decode --

CASES = [
    # dtype, D, BS, H, Hkv
    ("f32", 64, 16, 4, 4),
    ("f32", 128, 16, 8, 2),
    ("f32", 64, 32, 12, 4),
    ("f32", 128, 32, 16, 1),
    ("bf16", 128, 16, 32, 32),
    ("bf16", 128, 16, 32, 8),
    ("bf16", 128, 16, 64, 8),
    ("bf16", 64, 16, 8, 4),
    ("bf16", 64, 32, 12, 4),
    ("bf16", 128, 32, 16, 1),
    ("bf16", 128, 16, 6, 2),
    # groups above 8 on CUDA cores are split over two CTAs of one kv head
    ("f32", 64, 16, 12, 1),
    ("f32", 128, 16, 10, 1),
    ("bf16", 128, 16, 12, 1),
    # fp32 groups above 4 take TF32 tensor-core tiles by default
    ("f32", 128, 16, 12, 2),
    ("f32", 64, 16, 8, 1),
]


@pytest.mark.parametrize("partition", [-1, 0, 64])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
def test_decode_matches_oracle(case, partition):
    dtype, D, BS, H, Hkv = case
    w = _w(dtype, D, BS, H, Hkv, seed=CASES.index(case))
    ref, _, _ = oracle_after_write(w)
    paths = [pagedkv.PATH_AUTO, pagedkv.PATH_FMA, pagedkv.PATH_MMA]
    for path in paths:
        dw = run_decode(w, path=path, partition_tokens=partition)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, dtype, f"{case} path={path} partition={partition}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bf16_output(dtype):
    w = _w(dtype, 128, 16, 16, 4, seed=5)
    ref, _, _ = oracle_after_write(w)
    dw = run_decode(w, partition_tokens=128, out_dtype=torch.bfloat16)
    assert_close(dw.out, ref, dtype, "bf16 output")


def test_tiny_f32_workload():
    w = workload.make("tiny_f32")
    ref, _, _ = oracle_after_write(w)
    dw = run_decode(w)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "f32", "tiny_f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_long_context_many_partitions(dtype):
    w = _w(dtype, 128, 16, 16, 2, ctx=[9000, 4097, 1, 513], seed=9)
    ref, _, _ = oracle_after_write(w)
    for pt in (-1, 0, 512, 2048):
        dw = run_decode(w, partition_tokens=pt)
        assert_close(dw.out, ref, dtype, f"partition {pt}")


def test_random_shapes_sweep():
    rng = np.random.default_rng(77)
    for trial in range(12):
        dtype = ["f32", "bf16"][trial % 2]
        D = [64, 128][(trial // 2) % 2]
        BS = [16, 32][(trial // 4) % 2]
        Hkv = int(rng.integers(1, 5))
        G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        S = int(rng.integers(1, 9))
        ctx = rng.integers(0, 1500, size=S).tolist()
        w = _w(dtype, D, BS, Hkv * G, Hkv, ctx=ctx, seed=300 + trial)
        ref, _, _ = oracle_after_write(w)
        pt = int(rng.choice([-1, 0, BS * 4, BS * 16]))
        dw = run_decode(w, partition_tokens=pt)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, dtype, f"trial {trial}: {dtype} D{D} BS{BS} G{G} ctx {ctx} pt {pt}")


# ------------------------------------------------- blocks of 64 to 256 tokens

LARGE_BLOCK_CASES = [
    # dtype, D, BS, H, Hkv
    ("bf16", 128, 64, 32, 8),
    ("bf16", 128, 128, 8, 8),
    ("bf16", 64, 256, 16, 2),
    ("f32", 64, 64, 4, 4),
    ("f32", 128, 256, 8, 2),
]


@pytest.mark.parametrize("case", LARGE_BLOCK_CASES, ids=lambda c: "_".join(map(str, c)))
def test_large_blocks_match_oracle(case):
    """Blocks of 64, 128 and 256 tokens (the page's range of roughly 16 to
    256): the kernel stages each block in runs of 16 rows named by the
    block's one table entry; contexts end mid-run, mid-block, on a run and on
    a block boundary."""
    dtype, D, BS, H, Hkv = case
    ctx = [1, 31, 32, 33, BS - 1, BS, BS + 1, 3 * BS + 17, 1000]
    w = _w(dtype, D, BS, H, Hkv, ctx=ctx, seed=400 + LARGE_BLOCK_CASES.index(case))
    ref, _, _ = oracle_after_write(w)
    paths = [pagedkv.PATH_AUTO, pagedkv.PATH_FMA, pagedkv.PATH_MMA]
    for pt in (-1, 0, 2 * BS):
        for path in paths:
            dw = run_decode(w, path=path, partition_tokens=pt)
            assert pagedkv.get_device_error(dw.pool) == 0
            assert_close(dw.out, ref, dtype, f"{case} path={path} partition={pt}")


@pytest.mark.parametrize("BS", [64, 256])
def test_large_block_cache_write_bit_exact(BS):
    w = _w("bf16", 128, BS, 8, 4, ctx=[1, BS, BS + 1, 2 * BS + 5], seed=450)
    dw = pagedkv.DeviceWorkload(w)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, w.slot_mapping) == 0
    assert torch.equal(dw.k_pool.cpu().view(torch.int16), kp.view(torch.int16))
    assert torch.equal(dw.v_pool.cpu().view(torch.int16), vp.view(torch.int16))


def _reblock(w, BS):
    """The same logical tokens laid out in blocks of BS (sequential placement)."""
    S, Hkv, D = w.num_seqs, w.num_kv_heads, w.head_dim
    nblk = [-(-int(c) // BS) for c in w.context_lens]
    NB, MB = sum(nblk), max(nblk)
    k = torch.zeros((NB, Hkv, BS, D), dtype=w.k_pool.dtype)
    v = torch.zeros_like(k)
    bt = np.full((S, MB), -1, dtype=np.int32)
    nxt = 0
    for s in range(S):
        for b in range(nblk[s]):
            bt[s, b] = nxt
            for j in range(b * BS, min(int(w.context_lens[s]), (b + 1) * BS)):
                ob, orow = int(w.block_tables[s, j // w.block_size]), j % w.block_size
                k[nxt, :, j % BS] = w.k_pool[ob, :, orow]
                v[nxt, :, j % BS] = w.v_pool[ob, :, orow]
            nxt += 1
    slot = np.array([int(bt[s, (int(c) - 1) // BS]) * BS + (int(c) - 1) % BS
                     for s, c in enumerate(w.context_lens)], dtype=np.int64)
    return dataclasses.replace(w, block_size=BS, num_blocks=NB, max_blocks_per_seq=MB,
                               block_tables=bt, slot_mapping=slot, k_pool=k, v_pool=v)


def test_large_blocks_equal_small_blocks_bitwise():
    """The same tokens in blocks of 256 and of 32 give the same bits: the
    kernel's arithmetic runs over 16-row runs either way, in the same order."""
    w256 = _w("bf16", 128, 256, 32, 8, ctx=[5, 300, 777, 1024], seed=460)
    outs = []
    for w in (w256, _reblock(w256, 32)):
        dw = run_decode(w, partition_tokens=512)
        assert pagedkv.get_device_error(dw.pool) == 0
        outs.append(dw.out.cpu())
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))


# ------------------------------------------------------------- fp16 pools

F16_CASES = [
    # D, BS, H, Hkv
    (128, 16, 32, 32),
    (128, 16, 32, 8),
    (64, 32, 16, 2),
    (128, 64, 16, 4),
    (64, 16, 6, 2),
]


@pytest.mark.parametrize("case", F16_CASES, ids=lambda c: "_".join(map(str, c)))
def test_f16_decode_matches_oracle(case):
    """fp16 pools and queries: CUDA-core and fp16 tensor-core paths, whole
    and split contexts, against the oracle on the same fp16 values."""
    D, BS, H, Hkv = case
    w = _w("f16", D, BS, H, Hkv, seed=500 + F16_CASES.index(case))
    ref, _, _ = oracle_after_write(w)
    for pt in (-1, 0, 2 * BS):
        for path in (pagedkv.PATH_AUTO, pagedkv.PATH_FMA, pagedkv.PATH_MMA):
            dw = run_decode(w, path=path, partition_tokens=pt)
            assert pagedkv.get_device_error(dw.pool) == 0
            assert_close(dw.out, ref, "f16", f"{case} path={path} partition={pt}")


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_f16_output(dtype):
    """An fp16 output is the fp32 result rounded once to fp16."""
    w = _w(dtype, 128, 16, 16, 4, seed=520)
    ref, _, _ = oracle_after_write(w)
    dw16 = run_decode(w, partition_tokens=128, out_dtype=torch.float16)
    assert_close(dw16.out, ref, dtype, "fp16 output")
    dw32 = run_decode(w, partition_tokens=128, out_dtype=torch.float32)
    assert torch.equal(dw32.out.to(torch.float16).cpu().view(torch.int16),
                       dw16.out.cpu().view(torch.int16))


# ------------------------------------------------------------ head size 256

D256_CASES = [
    # dtype, BS, H, Hkv
    ("bf16", 16, 8, 8),
    ("bf16", 16, 16, 8),
    ("f16", 16, 16, 4),
    ("bf16", 64, 32, 4),
    ("f16", 32, 16, 1),
]


@pytest.mark.parametrize("case", D256_CASES, ids=lambda c: "_".join(map(str, c)))
def test_head_size_256_matches_oracle(case):
    """512-byte rows (16-bit pools): blocks are staged in runs of 16 rows;
    CUDA-core rows for groups up to 4 (larger groups forced onto CUDA cores
    are split over CTAs of 4 rows), tensor-core tiles otherwise."""
    dtype, BS, H, Hkv = case
    w = _w(dtype, 256, BS, H, Hkv, seed=600 + D256_CASES.index(case))
    ref, _, _ = oracle_after_write(w)
    paths = [pagedkv.PATH_AUTO, pagedkv.PATH_MMA, pagedkv.PATH_FMA]
    for pt in (-1, 0, 2 * BS):
        for path in paths:
            dw = run_decode(w, path=path, partition_tokens=pt)
            assert pagedkv.get_device_error(dw.pool) == 0
            assert_close(dw.out, ref, dtype, f"{case} path={path} partition={pt}")


def test_head_size_256_unsupported_combinations_are_refused():
    """fp32 pools are not built at head size 256; the call returns
    PKV_ERR_UNSUPPORTED and launches nothing."""
    w32 = _w("f32", 256, 16, 8, 8, ctx=[5, 40], seed=640)
    dw = pagedkv.DeviceWorkload(w32)
    with pytest.raises(pagedkv.PagedKVError) as e:
        dw.decode()
    assert e.value.status == pagedkv.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0


def test_random_shapes_sweep_wide():
    """Random shapes over every storage type, block sizes 16-256 and head
    sizes 64-256 (256 with 16-bit storage), against the oracle."""
    rng = np.random.default_rng(91)
    for trial in range(16):
        dtype = ["f32", "bf16", "f16"][trial % 3]
        D = int(rng.choice([64, 128] + ([256] if dtype != "f32" else [])))
        BS = int(rng.choice([16, 32, 64, 128, 256]))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 4, 5, 8] if D < 256 else [1, 2, 4, 8]))
        S = int(rng.integers(1, 7))
        ctx = rng.integers(0, 1300, size=S).tolist()
        w = _w(dtype, D, BS, Hkv * G, Hkv, ctx=ctx, seed=700 + trial)
        ref, _, _ = oracle_after_write(w)
        pt = int(rng.choice([-1, 0, BS * 2, BS * 4]))
        dw = run_decode(w, partition_tokens=pt)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, dtype, f"trial {trial}: {dtype} D{D} BS{BS} G{G} ctx {ctx} pt {pt}")


def test_largest_batch_of_sequences():
    """num_seqs at its bound (65535, the grid's y extent), short ragged
    contexts including empty ones; every sequence against the oracle."""
    S = 65535
    ctx = np.random.default_rng(77).integers(0, 41, size=S).tolist()
    w = _w("bf16", 64, 16, 4, 2, ctx=ctx, seed=880)
    ref, _, _ = oracle_after_write(w)
    dw = run_decode(w, partition_tokens=0)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", "65535 sequences")


def test_more_partitions_than_one_weight_chunk():
    """A 600k-token context in 512-token partitions (1172 parts) takes the
    many-part combine through more than one 1024-part chunk of weights."""
    w = _w("bf16", 64, 16, 4, 1, ctx=[600_000, 3, 70_000], seed=890)
    ref, _, _ = oracle_after_write(w)
    dw = run_decode(w, partition_tokens=512)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", "1172 partitions")
