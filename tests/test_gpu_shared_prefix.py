"""The shared-prefix decode (pkv_paged_attention_decode_shared_prefix) against
the float64 oracle.

Sequences forked from one prompt share the prompt's physical blocks (the
Hacker News thread on PagedAttention; Qualiteg's per-sequence block tables):
the attention result is the same as for private copies, which the oracle
computes by gathering each sequence's blocks through its own table.  The
cases cover ragged groups, every GQA group size the kernel packs (1 to 16
query heads per KV head, with members split across 32-row work items),
empty suffixes, partial last blocks, head sizes 64, 128 and 256, block sizes
16 to 256, both output types, and group descriptions that break the rules (reported in the
error word; the output must still be exact).
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


def _w(name, ctx, groups, H, Hkv, D=128, BS=16, seed=0, **kw):
    return workload.build(name, dtype="bf16", context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                          head_dim=D, block_size=BS, data_seed=5000 + seed,
                          meta_seed=6000 + seed, groups=groups, **kw)


def _run(w, partition=0, out_dtype=torch.float32, **setup):
    dw = pagedkv.DeviceWorkload(w, out_dtype=out_dtype)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    dw.shared_prefix_setup(partition_tokens=partition, **setup)
    dw.decode_shared_prefix()
    torch.cuda.synchronize()
    return dw


def _prefix_ctx(prefix, suffixes):
    return [prefix + s for s in suffixes]


def _varied_groups(n_groups=70, seed=2024):
    """More groups than the planning CTA has warps: one to four members each,
    prefixes of 0 to 5 whole blocks, every member with at least one own token
    (so no two members write into a shared block)."""
    rng = np.random.default_rng(seed)
    ctx, groups = [], []
    for _ in range(n_groups):
        m = int(rng.choice([1, 1, 2, 3, 4]))
        pre = int(rng.choice([0, 16, 32, 64, 80]))
        ctx += [pre + int(x) for x in rng.integers(1, 150, size=m)]
        groups.append((m, pre))
    return ctx, groups


CASES = {
    # name: (context lengths, groups, H, Hkv, D, BS)
    "g4_eight_members": (_prefix_ctx(256, [0, 1, 15, 16, 17, 100, 300, 700]), [(8, 256)],
                         32, 8, 128, 16),
    "g4_ragged_groups": ([70, 64, 100, 5, 130, 128, 300, 129, 200, 40, 33],
                         [(3, 64), (1, 0), (5, 128), (2, 32)], 16, 4, 128, 16),
    "mha_g1": (_prefix_ctx(512, [3, 40, 90, 0, 17, 600]), [(6, 512)], 8, 8, 128, 16),
    "g8_two_items": (_prefix_ctx(320, [1, 2, 3, 50, 60, 200]), [(6, 320)], 64, 8, 128, 16),
    "g16_pairs": (_prefix_ctx(160, [9, 0, 31]), [(3, 160)], 16, 1, 128, 16),
    "g3_odd": (_prefix_ctx(96, list(range(0, 130, 13))), [(10, 96)], 6, 2, 128, 16),
    "d64_bs32": (_prefix_ctx(384, [5, 64, 33, 1]), [(2, 384), (2, 96)], 8, 2, 64, 32),
    "d128_bs32": (_prefix_ctx(640, [31, 32, 33, 500]), [(4, 640)], 16, 4, 128, 32),
    "d64_bs16_mha": (_prefix_ctx(48, [1, 2, 3]), [(3, 48)], 4, 4, 64, 16),
    "big_group": (_prefix_ctx(1024, list(range(1, 40 * 7, 7))), [(40, 1024)], 8, 8, 128, 16),
    "varied_groups": (*_varied_groups(), 8, 2, 128, 16),
    # 256-wide heads: one 16-row tile per item (16 / G members)
    "d256_g4": (_prefix_ctx(256, [0, 1, 17, 100, 300]), [(5, 256)], 16, 4, 256, 16),
    "d256_g8_bs64": (_prefix_ctx(128, [3, 64, 65]), [(3, 128)], 16, 2, 256, 64),
    "d256_g1_mha": (_prefix_ctx(96, list(range(1, 120, 7))), [(17, 96)], 4, 4, 256, 16),
}


@pytest.mark.parametrize("partition", [0, -1, 64])
@pytest.mark.parametrize("case", sorted(CASES))
def test_shared_prefix_matches_oracle(case, partition):
    ctx, groups, H, Hkv, D, BS = CASES[case]
    if partition > 0 and partition % BS:
        partition = BS * 4
    w = _w(case, ctx, groups, H, Hkv, D, BS, seed=sorted(CASES).index(case))
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, partition)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", f"{case} partition {partition}")


@pytest.mark.parametrize("case", ["g4_eight_members", "g4_ragged_groups", "d64_bs32", "d256_g8_bs64"])
def test_shared_prefix_bf16_output(case):
    ctx, groups, H, Hkv, D, BS = CASES[case]
    w = _w(case, ctx, groups, H, Hkv, D, BS, seed=3)
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, 0, torch.bfloat16)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", f"{case} bf16 output")


def test_no_sharing_and_empty_contexts():
    """Groups of one (nothing shared), including zero-length contexts."""
    ctx = [0, 1, 17, 0, 900, 2048, 5]
    w = _w("flat", ctx, [(1, 0)] * len(ctx), 32, 8, seed=11)
    ref, _, _ = oracle_after_write(w)
    for pt in (0, 256, -1):
        dw = _run(w, pt)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, "bf16", f"flat partition {pt}")
    assert float(dw.out[0].abs().max()) == 0.0 and float(dw.out[3].abs().max()) == 0.0


def test_repeat_calls_are_bitwise_equal():
    ctx, groups, H, Hkv, D, BS = CASES["g4_ragged_groups"]
    w = _w("rep", ctx, groups, H, Hkv, D, BS, seed=12)
    dw = _run(w, 64)
    first = dw.out.clone()
    for _ in range(3):
        dw.decode_shared_prefix()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int32), dw.out.view(torch.int32))


def test_agrees_with_the_plain_decode():
    ctx, groups, H, Hkv, D, BS = CASES["g8_two_items"]
    w = _w("plain", ctx, groups, H, Hkv, D, BS, seed=13)
    sp = _run(w, 0)
    plain = pagedkv.DeviceWorkload(w)
    plain.step()
    torch.cuda.synchronize()
    assert float((sp.out - plain.out).abs().max()) <= 4e-3


# ------------------------------------------------ broken group descriptions

def _broken(setup, expect_exact=True):
    ctx = _prefix_ctx(256, [20, 30, 300, 5, 0, 64])
    w = _w("broken", ctx, [(3, 256), (3, 256)], 16, 4, seed=14)
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, 0, **setup)
    bits = pagedkv.get_device_error(dw.pool)
    assert bits & pagedkv.FAULT_PREFIX, bits
    if expect_exact:
        assert_close(dw.out, ref, "bf16", f"fallback after {setup}")


def test_group_starts_not_covering_the_batch():
    _broken(dict(group_starts=[0, 4, 3, 6], prefix_lens=[256, 256, 0]))
    _broken(dict(group_starts=[0, 3, 5], prefix_lens=[256, 256]))


def test_prefix_longer_than_a_member():
    _broken(dict(prefix_lens=[256, 512], max_prefix_len=512))


def test_prefix_not_whole_blocks():
    _broken(dict(prefix_lens=[250, 256]))


def test_prefix_above_host_bound():
    _broken(dict(prefix_lens=[256, 256], max_prefix_len=128))


def test_prefix_negative():
    _broken(dict(prefix_lens=[-16, 256]))


def test_tables_that_differ_inside_the_prefix_are_reported():
    # members share 256 tokens, the description claims 272 (one block more)
    _broken(dict(prefix_lens=[272, 256], max_prefix_len=272), expect_exact=False)


# The full-size shared-prefix workload (256 sequences, 32 groups of 8) is
# compared with the oracle on every sequence in test_gpu_fullsize.py.


# ---------------------------------------------------- plan once, run per layer

def test_one_plan_serves_several_layers():
    """A model's layers share the step's batch: plan once, run per layer with
    that layer's queries (here: the same pool, new queries each time)."""
    ctx, groups, H, Hkv, D, BS = CASES["g4_ragged_groups"]
    w = _w("layers", ctx, groups, H, Hkv, D, BS, seed=21)
    dw = pagedkv.DeviceWorkload(w)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    dw.shared_prefix_setup(partition_tokens=64)
    dw.shared_prefix_plan()
    g = torch.Generator().manual_seed(5)
    for layer in range(4):
        q = torch.randn(w.q.shape, generator=g).to(torch.bfloat16)
        dw.q.copy_(q)
        dw.decode_shared_prefix_run()
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        w.q = q
        ref, _, _ = oracle_after_write(w)
        assert_close(dw.out, ref, "bf16", f"layer {layer}")


def test_run_without_or_against_another_plan_is_reported():
    ctx, groups, H, Hkv, D, BS = CASES["g4_eight_members"]
    w = _w("noplan", ctx, groups, H, Hkv, D, BS, seed=22)
    dw = pagedkv.DeviceWorkload(w)
    dw.shared_prefix_setup(partition_tokens=0)
    dw.sp_workspace.zero_()
    dw.out.fill_(7.0)
    dw.decode_shared_prefix_run()  # no plan in the workspace
    assert pagedkv.get_device_error(dw.pool) & pagedkv.FAULT_PREFIX
    assert float(dw.out.min()) == 7.0 == float(dw.out.max())  # nothing written
    dw.shared_prefix_plan()
    dw.sp_partition = -1  # a run with another geometry than the plan's (fits the workspace)
    dw.decode_shared_prefix_run()
    assert pagedkv.get_device_error(dw.pool) & pagedkv.FAULT_PREFIX



@pytest.mark.parametrize("plan_dtype,plan_d,run_dtype,run_d", [
    ("bf16", 128, "bf16", 64),   # 32 query rows per item against a kernel of 16
    ("bf16", 128, "f32", 128),   # the same head size, fp32 storage: 16 rows per item
    ("bf16", 64, "bf16", 128),
])
def test_run_against_a_plan_for_another_pool_is_reported(plan_dtype, plan_d, run_dtype, run_d):
    """A plan records the members its prefix items hold, which follow the
    pool's head size and storage type; a run with a pool of other rows per
    item writes nothing and reports the plan as not its own."""
    ctx, groups, H, Hkv, D, BS = CASES["g4_eight_members"]
    mk = lambda name, dt, d: workload.build(  # noqa: E731
        name, dtype=dt, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=d,
        block_size=BS, data_seed=5023, meta_seed=6023, groups=groups)
    dp = pagedkv.DeviceWorkload(mk("plan", plan_dtype, plan_d))
    dp.shared_prefix_setup(partition_tokens=0)
    dr = pagedkv.DeviceWorkload(mk("run", run_dtype, run_d))
    dr.shared_prefix_setup(partition_tokens=0)
    ws = torch.zeros(max(dp.sp_workspace.numel(), dr.sp_workspace.numel()), dtype=torch.uint8,
                     device=dp.sp_workspace.device)
    dp.sp_workspace = ws
    dr.sp_workspace = ws
    dp.shared_prefix_plan()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dp.pool) == 0
    dr.out.fill_(7.0)
    dr.decode_shared_prefix_run()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dr.pool) & pagedkv.FAULT_PREFIX
    assert float(dr.out.min()) == 7.0 == float(dr.out.max())  # nothing written


# ------------------------------------------------------------ the work list

def _expected_items(w, pbp, pbs):
    """Work items of the group description, derived on the host: per group
    with a shared prefix, ceil(members / floor(R / G)) row sets x the prefix
    parts (R = 32 query rows per item for a 128-wide head, 16 otherwise); per
    sequence, its own blocks after the prefix in parts of pbs."""
    BS, G = w.block_size, w.num_heads // w.num_kv_heads
    mpi = (32 if w.head_dim == 128 else 16) // G
    gs, gp = w.groups()
    ctx = np.asarray(w.context_lens)
    pre, suf = [], []
    for i in range(len(gp)):
        start, end = int(gs[i]), int(gs[i + 1])
        pblk = int(gp[i]) // BS if end - start >= 2 else 0
        pp = -(-pblk // pbp)
        for m0 in range(start, end, mpi):
            for q in range(pp):
                b0, b1 = q * pbp, min(pblk, (q + 1) * pbp)
                pre.append((m0, min(mpi, end - m0), start, b0, b1, q, b1 * BS))
        for s in range(start, end):
            nb = -(-int(ctx[s]) // BS)
            for k, b0 in enumerate(range(pblk, nb, pbs)):
                suf.append((s, 1, s, b0, min(nb, b0 + pbs), pp + k, int(ctx[s])))
    return pre, suf


@pytest.mark.parametrize("case", ["g4_ragged_groups", "big_group", "g3_odd", "varied_groups"])
def test_plan_lists_every_item_once_largest_first(case):
    """The plan's entries are exactly the items of the description, each
    region (prefix items, then suffix items) in non-increasing block count, so
    the persistent grid's last items are its shortest."""
    ctx, groups, H, Hkv, D, BS = CASES[case]
    w = _w(case, ctx, groups, H, Hkv, D, BS, seed=31)
    dw = pagedkv.DeviceWorkload(w)
    dw.shared_prefix_setup(partition_tokens=64)
    dw.shared_prefix_plan()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    ws = dw.sp_workspace.cpu().numpy().view(np.int32)
    S = w.num_seqs
    r = lambda x: -(-x // 256) * 256  # noqa: E731
    off_entries = (256 + r(S * 4) + r(S * 8)) // 4
    pbp = pbs = 64 // BS
    pp = -(-min(dw.max_prefix_len, dw.max_context_len) // 64)
    n_pre, n_suf = int(ws[0]), int(ws[1])
    ent = ws[off_entries:].reshape(-1, 8)
    got_pre = [tuple(int(x) for x in e[:7]) for e in ent[:n_pre]]
    got_suf = [tuple(int(x) for x in e[:7]) for e in ent[S * pp:S * pp + n_suf]]
    exp_pre, exp_suf = _expected_items(w, pbp, pbs)
    assert sorted(got_pre) == sorted(exp_pre)
    assert sorted(got_suf) == sorted(exp_suf)
    for got in (got_pre, got_suf):
        sizes = [e[4] - e[3] for e in got]
        assert sizes == sorted(sizes, reverse=True), sizes
    # partial counts: prefix parts plus own parts of every sequence
    nparts = ws[64:64 + S]
    for s in range(S):
        assert nparts[s] == sum(1 for e in exp_pre if e[0] <= s < e[0] + e[1]) + \
            sum(1 for e in exp_suf if e[0] == s)


# ----------------------------------------------- blocks of 64 to 256 tokens

@pytest.mark.parametrize("BS", [64, 128, 256])
def test_shared_prefix_large_blocks(BS):
    """Blocks above 16 tokens are listed and staged as 16-row runs; the
    prefix stays whole blocks and the combine checks the tables per block."""
    ctx = _prefix_ctx(2 * BS, [0, 1, 31, 33, BS, BS + 7, 3 * BS])
    groups = [(4, 2 * BS), (3, BS)]
    w = _w(f"large{BS}", ctx, groups, 32, 8, 128, BS, seed=40 + BS // 64)
    ref, _, _ = oracle_after_write(w)
    for pt in (0, -1, BS):
        dw = _run(w, pt)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, "bf16", f"BS {BS} partition {pt}")


def test_shared_prefix_large_block_tables_that_differ_are_reported():
    """Member 2 names its own third block where the group shares block 1:
    the combine compares the tables per block (not per run) and reports it."""
    BS = 64
    ctx = _prefix_ctx(2 * BS, [10, 20, 30])
    w = _w("large_bad", ctx, [(3, 2 * BS)], 16, 4, 128, BS, seed=47)
    bt = w.block_tables.copy()
    assert bt[2, 2] >= 0 and bt[2, 2] != bt[0, 1]
    bt[2, 1] = bt[2, 2]
    w.block_tables = bt
    dw = _run(w, 0)
    assert pagedkv.get_device_error(dw.pool) & pagedkv.FAULT_PREFIX


# ------------------------------------------------------------- fp16 pools

@pytest.mark.parametrize("case", ["g4_ragged_groups", "g8_two_items", "d64_bs32", "d256_g4"])
def test_shared_prefix_f16(case):
    ctx, groups, H, Hkv, D, BS = CASES[case]
    w = workload.build(case, dtype="f16", context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                       head_dim=D, block_size=BS, data_seed=5300, meta_seed=6300, groups=groups)
    ref, _, _ = oracle_after_write(w)
    for out_dtype in (torch.float32, torch.float16):
        dw = _run(w, 0, out_dtype)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, "f16", f"{case} fp16 pools, out {out_dtype}")


# ------------------------------------------------------------- fp32 pools

@pytest.mark.parametrize("case", ["g4_eight_members", "g4_ragged_groups", "mha_g1", "g8_two_items",
                                  "g16_pairs", "g3_odd", "d64_bs32", "big_group", "varied_groups"])
def test_shared_prefix_f32(case):
    """fp32 pools: TF32 tiles of 16 query rows, every product as three TF32
    products, held to the fp32 tolerance of 1e-5."""
    ctx, groups, H, Hkv, D, BS = CASES[case]
    w = workload.build(case, dtype="f32", context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                       head_dim=D, block_size=BS, data_seed=5500, meta_seed=6500, groups=groups)
    ref, _, _ = oracle_after_write(w)
    for partition in (0, -1, 64):
        for out_dtype in (torch.float32, torch.bfloat16):
            dw = _run(w, partition, out_dtype)
            assert pagedkv.get_device_error(dw.pool) == 0
            assert_close(dw.out, ref, "f32", f"{case} fp32 pools, partition {partition}, out {out_dtype}")


# ------------------------------------------------------------ random sweep

def test_shared_prefix_random_sweep():
    """Random group structures, prefix lengths, contexts, partitions, block
    and head sizes, group sizes and storage types, each against the oracle."""
    rng = np.random.default_rng(2024)
    for trial in range(14):
        BS = int(rng.choice([16, 32, 64]))
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
        dtype = ["bf16", "f16"][trial % 2]
        groups, ctx = [], []
        for _ in range(int(rng.integers(1, 5))):
            members = int(rng.integers(1, 12))
            prefix = BS * int(rng.integers(0, 6)) if members > 1 else 0
            groups.append((members, prefix))
            # at most one member ends on the prefix: its new token is written
            # into the shared block, and two such writers would race on a slot
            own = [int(rng.integers(1, 300)) for _ in range(members)]
            own[0] = int(rng.integers(0, 300))
            ctx += [prefix + o for o in own]
        w = workload.build(f"sweep{trial}", dtype=dtype, context_lens=ctx, num_heads=Hkv * G,
                           num_kv_heads=Hkv, head_dim=D, block_size=BS, data_seed=9000 + trial,
                           meta_seed=9100 + trial, groups=groups)
        ref, _, _ = oracle_after_write(w)
        pt = int(rng.choice([0, -1, BS, 4 * BS]))
        dw = _run(w, pt)
        assert pagedkv.get_device_error(dw.pool) == 0, trial
        assert_close(dw.out, ref, dtype, f"trial {trial}: BS{BS} D{D} G{G} groups {groups} pt {pt}")



@pytest.mark.parametrize("D,dtype,G", [(128, "bf16", 4), (256, "bf16", 4), (64, "f16", 8),
                                       (128, "f32", 4)])
def test_shared_prefix_automatic_parts_on_irregular_batches(D, dtype, G):
    """Batches large enough that the plan takes its longer automatic prefix
    parts (1024 or 2048 tokens), with irregular groups: one to sixteen
    members, prefixes of any whole number of blocks (so a prefix's last part
    is ragged) and own lengths from nothing to 700 tokens.  Every sequence
    is checked against the oracle, and the plan's prefix items are longer
    than the shortest candidate (512 tokens)."""
    rng = np.random.default_rng(77 + D + (1 if dtype == "f32" else 0))
    BS, Hkv = 16, 8
    groups, ctx = [], []
    while len(ctx) < 320:
        members = int(rng.integers(1, 17))
        prefix = BS * int(rng.integers(64, 400)) if members > 1 else 0
        groups.append((members, prefix))
        # at most one member ends on the prefix (two would write one shared slot)
        own = [int(rng.integers(1, 700)) for _ in range(members)]
        own[0] = int(rng.integers(0, 700))
        ctx += [prefix + o for o in own]
    w = workload.build(f"autoparts{D}{dtype}", dtype=dtype, context_lens=ctx, num_heads=Hkv * G,
                       num_kv_heads=Hkv, head_dim=D, block_size=BS, data_seed=9300 + D,
                       meta_seed=9400 + D, groups=groups)
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, 0, out_dtype=torch.bfloat16)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, dtype, f"D{D} {dtype} G{G}: {len(groups)} groups, automatic parts")
    ws = dw.sp_workspace.cpu().numpy().view(np.int32)
    S = w.num_seqs
    r = lambda x: -(-x // 256) * 256  # noqa: E731
    ent = ws[(256 + r(S * 4) + r(S * 8)) // 4:].reshape(-1, 8)[:int(ws[0])]
    assert int((ent[:, 4] - ent[:, 3]).max()) > 32, "the plan kept the shortest prefix parts"


def test_shared_prefix_random_sweep_d256():
    """The same sweep for 256-wide heads (items of 16 rows: 16 / G members)."""
    rng = np.random.default_rng(2256)
    for trial in range(6):
        BS = int(rng.choice([16, 32, 64]))
        Hkv = int(rng.integers(1, 3))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        dtype = ["bf16", "f16"][trial % 2]
        groups, ctx = [], []
        for _ in range(int(rng.integers(1, 4))):
            members = int(rng.integers(1, 10))
            prefix = BS * int(rng.integers(0, 5)) if members > 1 else 0
            groups.append((members, prefix))
            own = [int(rng.integers(1, 250)) for _ in range(members)]
            own[0] = int(rng.integers(0, 250))
            ctx += [prefix + o for o in own]
        w = workload.build(f"sweep256_{trial}", dtype=dtype, context_lens=ctx, num_heads=Hkv * G,
                           num_kv_heads=Hkv, head_dim=256, block_size=BS, data_seed=9300 + trial,
                           meta_seed=9400 + trial, groups=groups)
        ref, _, _ = oracle_after_write(w)
        pt = int(rng.choice([0, -1, BS, 4 * BS]))
        dw = _run(w, pt)
        assert pagedkv.get_device_error(dw.pool) == 0, trial
        assert_close(dw.out, ref, dtype, f"trial {trial}: BS{BS} G{G} groups {groups} pt {pt}")


def test_more_sequences_than_the_plan_stages():
    """Above 8192 sequences the planning kernel reads context lengths from
    global memory instead of staging them in shared memory."""
    rng = np.random.default_rng(31)
    groups, ctx = [], []
    while len(ctx) < 9000:
        members = int(rng.integers(1, 5))
        prefix = 16 * int(rng.integers(1, 4)) if members > 1 else 0
        groups.append((members, prefix))
        # every member's new token lies past the shared prefix (two members
        # ending on the prefix would write the same shared slot)
        ctx += [prefix + int(rng.integers(1, 40)) for _ in range(members)]
    w = workload.build("many", dtype="bf16", context_lens=ctx, num_heads=8, num_kv_heads=2,
                       head_dim=64, block_size=16, data_seed=4242, meta_seed=4343, groups=groups)
    assert w.num_seqs > 8192
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, 0)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", f"{w.num_seqs} sequences")


def test_more_than_32_parts_per_sequence():
    """A 4096-token prefix in 64-token parts gives every member more than 32
    partials: the combine walks its weights 32 at a time."""
    ctx = _prefix_ctx(4096, [1, 50, 700, 1500])
    w = _w("many_parts", ctx, [(4, 4096)], 16, 4, 128, 16, seed=77)
    ref, _, _ = oracle_after_write(w)
    dw = _run(w, 64)
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, "bf16", "64-token parts")


# --------------------------------------------------------- climbing scores

def _climbing_keys(w, rate):
    """Scale each stored key row by 1 + rate * (its logical position), once
    per physical block, and each new key by the factor of its position, so a
    row's scores climb along the context: the running maximum moves many times
    inside one work item, and many weights land just below the largest
    stale-reference weight the kernel lets through before it rescales."""
    BS = w.block_size
    k = w.k_pool.float()
    done = set()
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        for b in range(-(-c // BS)):
            pb = int(w.block_tables[s, b])
            if pb in done:
                continue
            done.add(pb)
            f = 1.0 + rate * (b * BS + torch.arange(BS, dtype=torch.float32))
            k[pb] *= f[None, :, None]
    w.k_pool = k.to(w.torch_dtype)
    f_new = 1.0 + rate * (torch.from_numpy(w.context_lens.astype(np.float32)) - 1.0)
    w.new_key = (w.new_key.float() * f_new[:, None, None]).to(w.torch_dtype)
    return w


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("case", ["g4_eight_members", "g8_two_items", "d64_bs32", "d256_g4",
                                  "big_group", "varied_groups"])
def test_shared_prefix_climbing_scores(case, dtype):
    ctx, groups, H, Hkv, D, BS = CASES[case]
    if dtype == "f32" and D > 128:
        pytest.skip("fp32 pools are built up to head size 128")
    w = workload.build(case, dtype=dtype, context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                       head_dim=D, block_size=BS, data_seed=5600, meta_seed=6600, groups=groups)
    # fp32 climbs half as steeply: at the full rate the scores reach ~120 in
    # log2 units, where the fp32 rounding of the scores alone (measured on the
    # CUDA-core path, which accumulates exactly in fp32) is at the 1e-5 tolerance
    _climbing_keys(w, rate=(10.0 if dtype == "f32" else 20.0) / max(ctx))
    ref, _, _ = oracle_after_write(w)
    for partition in (0, 64):
        dw = _run(w, partition)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, dtype, f"{case} {dtype} climbing scores, partition {partition}")
    # the plain decode on the same keys
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.float32)
    dw.step()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, dtype, f"{case} {dtype} climbing scores, plain decode")


# ------------------------------------------- faults and short items, all rings

@pytest.mark.parametrize("D", [64, 128, 256])
def test_shared_prefix_bad_block_id_sets_fault_and_spares_other_sequences(D):
    """A block id outside the pool in one member's own blocks: the kernel's
    bound check reports it and skips the block (for a 256-wide head the K and
    V halves of its one-stage ring are released separately); every sequence
    that does not name the block is still exact."""
    ctx = _prefix_ctx(64, [40, 70, 5, 100])
    w = _w(f"badblk{D}", ctx, [(4, 64)], 16, 4, D, 16, seed=900 + D)
    ref, _, _ = oracle_after_write(w)
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.float32)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    bt = w.block_tables
    bad_seq, bad_blk = 1, 5  # past the 4-block prefix: sequence 1's own block
    assert bt[bad_seq, bad_blk] >= 0 and not np.any(np.delete(bt, bad_seq, 0) == bt[bad_seq, bad_blk])
    dw.block_tables[bad_seq, bad_blk] = w.num_blocks + 7
    dw.shared_prefix_setup()
    dw.decode_shared_prefix()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == pagedkv.FAULT_BLOCK_ID
    out = dw.out.cpu()
    assert torch.isfinite(out).all()
    for s in range(w.num_seqs):
        if s != bad_seq:
            assert_close(out[s], ref[s], "bf16", f"D{D}: unaffected sequence {s}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_shared_prefix_many_short_items(D):
    """Only items of one to three blocks, many per warp: each item is shorter
    than the lead the next item's claim needs, so the next item's first stages
    are requested after the current one's loop, item after item."""
    rng = np.random.default_rng(77 + D)
    groups, ctx = [], []
    for _ in range(150):
        members = int(rng.integers(1, 4))
        prefix = 16 * int(rng.integers(1, 3)) if members > 1 else 0
        groups.append((members, prefix))
        ctx += [prefix + int(rng.integers(1, 48)) for _ in range(members)]
    w = workload.build(f"short{D}", dtype="bf16", context_lens=ctx, num_heads=8, num_kv_heads=2,
                       head_dim=D, block_size=16, data_seed=7700 + D, meta_seed=7800 + D,
                       groups=groups)
    ref, _, _ = oracle_after_write(w)
    for partition in (0, 16):
        dw = _run(w, partition)
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, "bf16", f"D{D} short items, partition {partition}")
