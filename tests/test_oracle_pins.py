"""Pins for the float64 oracle: hand-derived fixtures, closed forms, brute
force and the invariants that the PagedAttention pages fix.

Every test here runs on the CPU.  Each pin targets a plausible mistake:
a wrong gather index, a transposed pool axis, an interleaved GQA mapping, a
dropped scale, a softmax of the wrong sign, a missing normalisation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_249_gb300 import workload
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- fixtures --

@pytest.mark.parametrize("name", ["paged_gather_uniform.json", "paged_two_token_softmax.json",
                                  "paged_gqa_grouping.json"])
def test_golden_paged_decode(name):
    g = _load(name)
    q = torch.tensor(g["query"], dtype=torch.float32)
    kp = torch.tensor(g["k_pool"], dtype=torch.float32)
    vp = torch.tensor(g["v_pool"], dtype=torch.float32)
    out = oracle.paged_decode(q, kp, vp, np.array(g["block_tables"]), np.array(g["context_lens"]),
                              g["scale"], num_threads=2)
    np.testing.assert_allclose(out, np.array(g["expected"]), rtol=0, atol=g["tolerance"])


def test_golden_reshape_and_cache():
    g = _load("reshape_tiny.json")
    shape = (g["num_blocks"], g["num_kv_heads"], g["block_size"], g["head_dim"])
    kp = torch.zeros(shape)
    vp = torch.zeros(shape)
    faults = oracle.reshape_and_cache(kp, vp, torch.tensor(g["key"], dtype=torch.float32),
                                      torch.tensor(g["value"], dtype=torch.float32),
                                      np.array(g["slot_mapping"]))
    assert faults == g["expected_faults"]
    assert torch.equal(kp, torch.tensor(g["expected_k_pool"], dtype=torch.float32))
    assert torch.equal(vp, torch.tensor(g["expected_v_pool"], dtype=torch.float32))


# ----------------------------------------------------------- closed forms --

def _single_seq(K, V, q, block_size=4, seed=0, dtype=torch.float32):
    """Place contiguous K/V rows [ctx][D] of one sequence into a shuffled pool."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    ctx, D = K.shape
    nblk = max(1, -(-ctx // block_size))
    NB = nblk + 3
    perm = np.random.default_rng(seed).permutation(NB)
    kp = torch.full((NB, 1, block_size, D), 7.0e3, dtype=torch.float64)
    vp = torch.full((NB, 1, block_size, D), -7.0e3, dtype=torch.float64)
    for j in range(ctx):
        kp[perm[j // block_size], 0, j % block_size] = torch.from_numpy(K[j])
        vp[perm[j // block_size], 0, j % block_size] = torch.from_numpy(V[j])
    bt = perm[:nblk].reshape(1, -1).astype(np.int32)
    qt = torch.tensor(np.asarray(q, dtype=np.float64)).reshape(1, 1, D)
    return qt.to(dtype), kp.to(dtype), vp.to(dtype), bt, np.array([ctx], dtype=np.int32)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(11)
    ctx, D = 37, 16
    k = rng.standard_normal(D)
    K = np.tile(k, (ctx, 1))
    V = rng.standard_normal((ctx, D))
    q = rng.standard_normal(D)
    args = _single_seq(K, V, q)
    out = oracle.paged_decode(*args, scale=0.3)[0, 0]
    Vs = args[2]  # compare against the float32-stored values
    Vf = np.array([Vs[args[3][0, j // 4], 0, j % 4].double().numpy() for j in range(ctx)])
    np.testing.assert_allclose(out, Vf.mean(axis=0), rtol=0, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(12)
    D = 8
    K = rng.standard_normal((1, D))
    V = rng.standard_normal((1, D)).astype(np.float32)
    out = oracle.paged_decode(*_single_seq(K, V, rng.standard_normal(D)), scale=2.0)[0, 0]
    assert np.array_equal(out, V[0].astype(np.float64))


def test_zero_scale_gives_mean_of_values():
    rng = np.random.default_rng(13)
    ctx, D = 21, 8
    K = rng.standard_normal((ctx, D)).astype(np.float32)
    V = rng.standard_normal((ctx, D)).astype(np.float32)
    out = oracle.paged_decode(*_single_seq(K, V, rng.standard_normal(D)), scale=0.0)[0, 0]
    np.testing.assert_allclose(out, V.astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)


@pytest.mark.parametrize("hot", [0, 5, 12])
def test_one_hot_key_closed_form(hot):
    """Only key `hot` is aligned with q: its score is scale*c*|q|^2, the rest 0.

    out = (e^z V_hot + sum_{i != hot} V_i) / (e^z + n - 1).  A flipped sign,
    a dropped scale or a wrong token index all break this.
    """
    rng = np.random.default_rng(14 + hot)
    ctx, D, c, scale = 13, 4, 0.75, 0.5
    q = np.array([1.0, -0.5, 0.25, 2.0])
    K = np.zeros((ctx, D))
    K[hot] = c * q
    V = rng.integers(-8, 9, size=(ctx, D)).astype(np.float64)
    z = scale * c * float(q @ q)
    expect = (math.exp(z) * V[hot] + (V.sum(axis=0) - V[hot])) / (math.exp(z) + ctx - 1)
    out = oracle.paged_decode(*_single_seq(K, V, q, dtype=torch.float32), scale=scale)[0, 0]
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


def test_two_keys_logistic_closed_form():
    q = np.array([0.5, 1.0])
    K = np.array([[1.0, -1.0], [2.0, 0.5]])
    V = np.array([[3.0, -2.0], [-1.0, 4.0]])
    scale = 0.75
    z0, z1 = scale * (q @ K[0]), scale * (q @ K[1])
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))
    expect = (1 - w1) * V[0] + w1 * V[1]
    out = oracle.paged_decode(*_single_seq(K, V, q), scale=scale)[0, 0]
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-14)


def test_empty_context_is_zero():
    w = workload.build("t", dtype="f32", context_lens=[0, 3], num_heads=2, num_kv_heads=1,
                       head_dim=8, block_size=4, data_seed=1, meta_seed=2)
    out = oracle.paged_decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_bad_block_id_is_rejected():
    w = workload.build("t", dtype="f32", context_lens=[9], num_heads=1, num_kv_heads=1,
                       head_dim=8, block_size=4, data_seed=1, meta_seed=2)
    bt = w.block_tables.copy()
    bt[0, 2] = w.num_blocks  # one past the pool
    with pytest.raises(ValueError):
        oracle.paged_decode(w.q, w.k_pool, w.v_pool, bt, w.context_lens, w.scale)


# -------------------------------------------------------------- brute force --

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("heads", [(4, 4), (4, 2), (8, 1)])
def test_matches_decimal_brute_force(dtype, heads):
    H, Hkv = heads
    ctx = [1, 6, 16, 17, 40]
    w = workload.build("brute", dtype=dtype, context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                       head_dim=8, block_size=4, data_seed=31, meta_seed=32, pool_blocks=26)
    out = oracle.paged_decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale,
                              num_threads=3)
    ref = _brute.paged_decode(w.q.float().numpy(), w.k_pool.float().numpy(),
                              w.v_pool.float().numpy(), w.block_tables, w.context_lens, w.scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


def test_tiny_f32_workload_matches_brute_force():
    w = workload.make("tiny_f32")
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, w.slot_mapping) == 0
    out = oracle.paged_decode(w.q, kp, vp, w.block_tables, w.context_lens, w.scale)
    ref = _brute.paged_decode(w.q.numpy(), kp.numpy(), vp.numpy(), w.block_tables,
                              w.context_lens, w.scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


# --------------------------------------------------------------- invariants --

def _contiguous_rows(pool, bt, s, g, ctx, BS):
    idx_b = [int(bt[s][j // BS]) for j in range(ctx)]
    idx_r = [j % BS for j in range(ctx)]
    return pool[idx_b, g, idx_r].double().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_paged_equals_contiguous_under_any_placement(dtype):
    """The block table is an indirection only: any physical placement of the
    same logical tokens gives the same result as contiguous K/V."""
    ctx = [3, 16, 31, 64, 100]
    outs = []
    for meta in (101, 202, 303):
        w = workload.build("perm", dtype=dtype, context_lens=ctx, num_heads=4, num_kv_heads=2,
                           head_dim=16, block_size=8, data_seed=5, meta_seed=meta,
                           pool_blocks=40)
        # the data is drawn per physical block; re-place it so that logical
        # token (s, pos) carries the same values for every placement
        base = workload.build("perm", dtype=dtype, context_lens=ctx, num_heads=4, num_kv_heads=2,
                              head_dim=16, block_size=8, data_seed=5, meta_seed=101,
                              pool_blocks=40)
        kp = torch.zeros_like(base.k_pool)
        vp = torch.zeros_like(base.v_pool)
        for s in range(w.num_seqs):
            for b in range(-(-ctx[s] // 8)):
                kp[w.block_tables[s, b]] = base.k_pool[base.block_tables[s, b]]
                vp[w.block_tables[s, b]] = base.v_pool[base.block_tables[s, b]]
        out = oracle.paged_decode(base.q, kp, vp, w.block_tables, w.context_lens, w.scale)
        outs.append(out)
        for s in range(w.num_seqs):
            for h in range(4):
                K = _contiguous_rows(kp, w.block_tables, s, h // 2, ctx[s], 8)
                V = _contiguous_rows(vp, w.block_tables, s, h // 2, ctx[s], 8)
                ref = oracle.attention_contiguous(base.q[s, h].double().numpy(), K, V, w.scale)
                assert np.array_equal(out[s, h], ref)
    # arithmetic order depends only on logical positions: bitwise equal
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_equals_unshared_copies():
    """Sequences whose tables point at the same prefix blocks give exactly the
    result of sequences holding private copies of those blocks."""
    ctx = [24 + 5, 24 + 9, 24 + 1, 24 + 16]
    w = workload.build("share", dtype="bf16", context_lens=ctx, num_heads=4, num_kv_heads=2,
                       head_dim=8, block_size=8, data_seed=7, meta_seed=8, group_size=2,
                       prefix_len=24)
    shared = oracle.paged_decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale)
    # private copies: append fresh blocks for the second member of each group
    kp, vp, bt = [w.k_pool], [w.v_pool], w.block_tables.copy()
    nb = w.num_blocks
    for s in range(1, w.num_seqs, 2):
        for b in range(3):
            kp.append(w.k_pool[bt[s, b]][None])
            vp.append(w.v_pool[bt[s, b]][None])
            bt[s, b] = nb
            nb += 1
    kp, vp = torch.cat(kp), torch.cat(vp)
    assert len(set(bt[:, :3].ravel().tolist())) == 12
    private = oracle.paged_decode(w.q, kp, vp, bt, w.context_lens, w.scale)
    assert np.array_equal(shared, private)


def test_token_order_and_shift_invariance():
    rng = np.random.default_rng(21)
    ctx, D = 29, 8
    q = rng.standard_normal(D)
    K = rng.standard_normal((ctx, D))
    V = rng.standard_normal((ctx, D))
    base = oracle.attention_contiguous(q, K, V, 0.4)
    perm = rng.permutation(ctx)
    np.testing.assert_allclose(oracle.attention_contiguous(q, K[perm], V[perm], 0.4), base,
                               rtol=0, atol=1e-13)
    # adding the same vector to every key shifts all scores equally
    shift = rng.standard_normal(D) * 3
    np.testing.assert_allclose(oracle.attention_contiguous(q, K + shift, V, 0.4), base,
                               rtol=0, atol=1e-12)


def test_linear_in_values_and_inside_their_hull():
    rng = np.random.default_rng(22)
    ctx, D = 19, 6
    q = rng.standard_normal(D)
    K = rng.standard_normal((ctx, D)) * 2
    V1 = rng.standard_normal((ctx, D))
    V2 = rng.standard_normal((ctx, D))
    o1 = oracle.attention_contiguous(q, K, V1, 1.0)
    o2 = oracle.attention_contiguous(q, K, V2, 1.0)
    o12 = oracle.attention_contiguous(q, K, 2.0 * V1 - 3.0 * V2, 1.0)
    np.testing.assert_allclose(o12, 2.0 * o1 - 3.0 * o2, rtol=0, atol=1e-13)
    assert np.all(o1 <= V1.max(axis=0) + 1e-15) and np.all(o1 >= V1.min(axis=0) - 1e-15)


def test_reshape_then_gather_round_trip_and_untouched_bytes():
    w = workload.make("tiny_f32")
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, w.slot_mapping) == 0
    touched = torch.zeros(w.num_blocks, w.block_size, dtype=torch.bool)
    for s in range(w.num_seqs):
        pos = int(w.context_lens[s]) - 1
        blk = int(w.block_tables[s, pos // w.block_size])
        assert torch.equal(kp[blk, :, pos % w.block_size], w.new_key[s])
        assert torch.equal(vp[blk, :, pos % w.block_size], w.new_value[s])
        touched[blk, pos % w.block_size] = True
    keep = ~touched[:, None, :, None].expand_as(kp)
    assert torch.equal(kp[keep], w.k_pool[keep]) and torch.equal(vp[keep], w.v_pool[keep])


def test_reshape_negative_slot_is_skipped_bf16():
    w = workload.build("neg", dtype="bf16", context_lens=[5, 9], num_heads=2, num_kv_heads=2,
                       head_dim=8, block_size=4, data_seed=3, meta_seed=4)
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    sm = w.slot_mapping.copy()
    sm[1] = -1
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, sm) == 0
    assert torch.equal(kp[sm[0] // 4, :, sm[0] % 4], w.new_key[0])
    blk, off = divmod(int(w.slot_mapping[1]), 4)
    assert torch.equal(kp[blk, :, off], w.k_pool[blk, :, off])


# ------------------------------------------------------------- fp16 input --

def test_fp16_storage_is_widened_exactly():
    """Every finite IEEE binary16 value, stored in a V pool, comes back from a
    one-token context bit for bit as the value the format defines (checked
    against numpy's own float16 conversion): sign, exponent bias, the
    implicit bit and the subnormals all enter the oracle exactly."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    vals = bits.view(np.float16)
    finite = vals[np.isfinite(vals)]
    D = 128
    rows = -(-finite.size // D)
    v = np.zeros(rows * D, dtype=np.float16)
    v[:finite.size] = finite
    vp = torch.from_numpy(v.reshape(rows, 1, 1, D).copy())  # one-token blocks, one kv head
    kp = torch.zeros_like(vp)
    q = torch.zeros(rows, 1, D, dtype=torch.float16)
    bt = np.arange(rows, dtype=np.int32).reshape(rows, 1)
    out = oracle.paged_decode(q, kp, vp, bt, np.ones(rows, dtype=np.int32), 1.0, num_threads=4)
    got = out.reshape(-1)[:finite.size]
    assert np.array_equal(got, finite.astype(np.float64))


def test_fp16_matches_brute_force():
    """A small fp16 batch against the pure-Python brute force on the same
    widened values."""
    w = workload.build("pin_f16", dtype="f16", context_lens=[1, 5, 17, 40], num_heads=4,
                       num_kv_heads=2, head_dim=64, block_size=16, data_seed=31, meta_seed=32)
    out = oracle.paged_decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.scale,
                              num_threads=2)
    ref = _brute.paged_decode(w.q.numpy(), w.k_pool.numpy(), w.v_pool.numpy(), w.block_tables,
                              w.context_lens, w.scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_block_size_does_not_change_the_result():
    """The same tokens laid out in blocks of 16, 64 and 256 tokens (the
    page's range of roughly 16 to 256) give bit-identical oracle outputs:
    paging is storage, not arithmetic."""
    w = workload.build("pin_bs", dtype="bf16", context_lens=[1, 255, 256, 257, 700],
                       num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, data_seed=61,
                       meta_seed=62)
    outs = []
    for BS in (16, 64, 256):
        S, Hkv, D = w.num_seqs, w.num_kv_heads, w.head_dim
        nblk = [-(-int(c) // BS) for c in w.context_lens]
        k = torch.zeros((sum(nblk), Hkv, BS, D), dtype=w.k_pool.dtype)
        v = torch.zeros_like(k)
        bt = np.full((S, max(nblk)), -1, dtype=np.int32)
        order = np.random.default_rng(BS).permutation(sum(nblk))  # scattered placement
        nxt = 0
        for s in range(S):
            for b in range(nblk[s]):
                bt[s, b] = order[nxt]
                for j in range(b * BS, min(int(w.context_lens[s]), (b + 1) * BS)):
                    src = int(w.block_tables[s, j // w.block_size]), j % w.block_size
                    k[order[nxt], :, j % BS] = w.k_pool[src[0], :, src[1]]
                    v[order[nxt], :, j % BS] = w.v_pool[src[0], :, src[1]]
                nxt += 1
        outs.append(oracle.paged_decode(w.q, k, v, bt, w.context_lens, w.scale, num_threads=2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
