"""A multi-step decode loop driven by the host block manager, on the GPU,
mirrored step by step on the host by the float64 oracle.

Each iteration: every live sequence grows by one token (the manager hands
out its slot, allocating or copying-on-write a shared block), pending block
copies run on the device (pkv_copy_blocks), the new K/V rows are written
(pkv_reshape_and_cache), the block tables are uploaded
(pkv_block_table_upload) and decode attention runs.  Sequences are forked
(shared prompt prefixes), finished and added along the way.  The device
pools must equal the host mirror byte for byte, and every step's attention
must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_249_gb300 import pagedkv
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,H,Hkv,BS", [("bf16", 16, 4, 16), ("f32", 8, 8, 32),
                                             ("f16", 16, 2, 64)])
def test_manager_driven_decode_loop(dtype, H, Hkv, BS):
    D, NB, MB = 128, 160, 24
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16}[dtype]
    gen = torch.Generator().manual_seed(1234)
    rnd = lambda *shape: torch.randn(*shape, generator=gen).to(tdt)  # noqa: E731

    k_dev = torch.empty(NB, Hkv, BS, D, dtype=tdt, device="cuda")
    v_dev = torch.empty_like(k_dev)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = pagedkv.BlockPool(k_dev, v_dev, err, zero_fill=True)
    k_host = torch.zeros(NB, Hkv, BS, D, dtype=tdt)
    v_host = torch.zeros_like(k_host)
    bm = pagedkv.BlockManager(NB, BS)
    scale = D ** -0.5

    def write(slots, keys, values):
        sm = np.asarray(slots, dtype=np.int64)
        assert oracle.reshape_and_cache(k_host, v_host, keys, values, sm) == 0
        pagedkv.reshape_and_cache(pool, keys.cuda(), values.cuda(), torch.from_numpy(sm).cuda())

    def copies():
        src, dst = bm.take_copies()
        if src.size:
            k_host[torch.from_numpy(dst).long()] = k_host[torch.from_numpy(src).long()]
            v_host[torch.from_numpy(dst).long()] = v_host[torch.from_numpy(src).long()]
            pagedkv.copy_blocks(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())

    live = []
    next_id = 0

    def add(n):
        nonlocal next_id
        slots = bm.add_sequence(next_id, n)
        write(slots, rnd(n, Hkv, D), rnd(n, Hkv, D))
        live.append(next_id)
        next_id += 1

    for n in (40, 100, 17, 250):
        add(n)
    for parent in (1, 3):
        bm.fork(parent, next_id)
        live.append(next_id)
        next_id += 1

    rng = np.random.default_rng(5)
    bt_dev = torch.empty(16, MB, dtype=torch.int32, device="cuda")
    for step in range(24):
        if step == 8:
            bm.free_sequence(live.pop(0))
        if step == 12:
            add(33)
            bm.fork(live[-1], next_id)
            live.append(next_id)
            next_id += 1
        slots = [bm.append_token(i) for i in live]
        copies()
        write(slots, rnd(len(live), Hkv, D), rnd(len(live), Hkv, D))
        bt_host, cl = bm.block_tables(live, MB)
        S = len(live)
        bt_pinned = torch.from_numpy(bt_host).pin_memory()
        pagedkv.block_table_upload(bt_dev[:S], bt_pinned, NB)
        q = rnd(S, H, D)
        out = torch.empty(S, H, D, dtype=torch.float32, device="cuda")
        max_ctx = int(cl.max())
        pt = int(rng.choice([-1, 0, 64]))
        ws = pagedkv.alloc_workspace(S, H, D, max_ctx, pt)
        pagedkv.paged_attention_decode(pool, out, q.cuda(), bt_dev[:S], torch.from_numpy(cl).cuda(),
                                       max_ctx, scale, partition_tokens=pt, workspace=ws)
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(pool) == 0
        ref = oracle.paged_decode(q, k_host, v_host, bt_host, cl, scale)
        assert_close(out, ref, dtype, f"step {step}")
    view = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(k_dev.cpu().view(view), k_host.view(view))
    assert torch.equal(v_dev.cpu().view(view), v_host.view(view))


def test_copy_blocks_bit_exact_and_faults():
    NB, Hkv, BS, D = 12, 2, 16, 64
    k = torch.randn(NB, Hkv, BS, D).to(torch.bfloat16).cuda()
    v = torch.randn(NB, Hkv, BS, D).to(torch.bfloat16).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = pagedkv.BlockPool(k, v, err)
    k0, v0 = k.cpu(), v.cpu()
    src = torch.tensor([3, 0, 7], dtype=torch.int32)
    dst = torch.tensor([5, 11, 1], dtype=torch.int32)
    pagedkv.copy_blocks(pool, src.cuda(), dst.cuda())
    assert pagedkv.get_device_error(pool) == 0
    ek, ev = k0.clone(), v0.clone()
    ek[dst.long()] = k0[src.long()]
    ev[dst.long()] = v0[src.long()]
    assert torch.equal(k.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(v.cpu().view(torch.int16), ev.view(torch.int16))
    pagedkv.copy_blocks(pool, torch.tensor([2, NB], dtype=torch.int32).cuda(),
                        torch.tensor([4, 6], dtype=torch.int32).cuda())
    assert pagedkv.get_device_error(pool) == pagedkv.FAULT_BLOCK_ID
    ek[4] = ek[2]
    ev[4] = ev[2]
    assert torch.equal(k.cpu().view(torch.int16), ek.view(torch.int16))  # block 6 untouched


def test_manager_driven_shared_prefix_decode_loop():
    """Parallel sampling through the block manager: prompts forked into
    families, every member grows by a token per step (copy-on-write of the
    shared partial block), and each step decodes with the shared-prefix path,
    its group description derived by the manager from the tables."""
    D, H, Hkv, BS, NB, MB = 128, 16, 4, 16, 256, 40
    tdt = torch.bfloat16
    gen = torch.Generator().manual_seed(99)
    rnd = lambda *shape: torch.randn(*shape, generator=gen).to(tdt)  # noqa: E731
    k_dev = torch.empty(NB, Hkv, BS, D, dtype=tdt, device="cuda")
    v_dev = torch.empty_like(k_dev)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = pagedkv.BlockPool(k_dev, v_dev, err, zero_fill=True)
    k_host = torch.zeros(NB, Hkv, BS, D, dtype=tdt)
    v_host = torch.zeros_like(k_host)
    bm = pagedkv.BlockManager(NB, BS)
    scale = D ** -0.5

    def write(slots, n):
        keys, values = rnd(n, Hkv, D), rnd(n, Hkv, D)
        sm = np.asarray(slots, dtype=np.int64)
        assert oracle.reshape_and_cache(k_host, v_host, keys, values, sm) == 0
        pagedkv.reshape_and_cache(pool, keys.cuda(), values.cuda(), torch.from_numpy(sm).cuda())

    def copies():
        src, dst = bm.take_copies()
        if src.size:
            k_host[torch.from_numpy(dst).long()] = k_host[torch.from_numpy(src).long()]
            v_host[torch.from_numpy(dst).long()] = v_host[torch.from_numpy(src).long()]
            pagedkv.copy_blocks(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())

    families = []  # lists of sequence ids, the prompt first
    next_id = 0
    for prompt, members in ((150, 4), (83, 3), (40, 1), (260, 2)):
        write(bm.add_sequence(next_id, prompt), prompt)
        fam = [next_id]
        next_id += 1
        for _ in range(members - 1):
            bm.fork(fam[0], next_id)
            fam.append(next_id)
            next_id += 1
        families.append(fam)

    bt_dev = torch.empty(16, MB, dtype=torch.int32, device="cuda")
    shared_seen = 0
    for step in range(12):
        live = [s for fam in families for s in fam]
        gs = np.cumsum([0] + [len(f) for f in families]).astype(np.int32)
        slots = [bm.append_token(s) for s in live]
        copies()
        write(slots, len(live))
        bt_host, cl = bm.block_tables(live, MB)
        prefix = bm.shared_prefix(live, gs)
        shared_seen += int((prefix > 0).sum())
        S = len(live)
        pagedkv.block_table_upload(bt_dev[:S], torch.from_numpy(bt_host).pin_memory(), NB)
        q = rnd(S, H, D)
        out = torch.empty(S, H, D, dtype=torch.float32, device="cuda")
        max_ctx, max_pre = int(cl.max()), int(prefix.max())
        ws = torch.empty(pagedkv.shared_prefix_workspace_bytes(S, H, D, max_ctx, max_pre),
                         dtype=torch.uint8, device="cuda")
        pagedkv.paged_attention_decode_shared_prefix(
            pool, out, q.cuda(), bt_dev[:S], torch.from_numpy(cl).cuda(), max_ctx, scale,
            torch.from_numpy(gs).cuda(), torch.from_numpy(prefix).cuda(), max_pre, ws)
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(pool) == 0
        ref = oracle.paged_decode(q, k_host, v_host, bt_host, cl, scale)
        assert_close(out, ref, "bf16", f"step {step}")
        if step == 6:  # one family member finishes
            bm.free_sequence(families[0].pop())
    assert shared_seen >= 3 * 12  # three families shared blocks every step
    assert torch.equal(k_dev.cpu().view(torch.int16), k_host.view(torch.int16))
