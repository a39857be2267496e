"""Seeded synthetic decode-step workloads for paged KV-cache attention.

This module only draws random numbers and lays out block tables; it holds
none of the attention arithmetic, so both the CUDA path and the float64
oracle can take their inputs from it.

Workload shapes follow the decode-step setting of the PagedAttention pages
(Qualiteg, "About PagedAttention for LLM serving": the section on logical
blocks, physical blocks and the block table, and point 1-2 under "[Regarding
Problem 1]" on splitting the KV cache into blocks): each running sequence owns a list
of fixed-size logical blocks mapped through a per-sequence block table onto
physical blocks of one shared pool, in no particular physical order.

Recipe (all draws from NumPy PCG64):
  * lengths and placement: ``PCG64(249100 + id)``; integers "uniform in
    [a, b]" are inclusive at both ends; physical placement is one
    ``permutation`` of the pool, handed out to logical blocks in
    sequence-major, block-minor order;
  * data: ``SeedSequence(249000 + id)`` spawns one child per tensor (q,
    K pool, V pool, new key, new value); each tensor is filled in chunks of
    2**24 float32 N(0,1) draws, chunk i from its own grandchild stream, so
    the values do not depend on the thread count;
  * bf16 (and fp16) workloads round those float32 draws to bf16 (fp16)
    with round-to-nearest-even (``torch.Tensor.to``); both sides see the
    rounded values.

Layout (our choice, 16-byte aligned rows): K pool and V pool are separate
``[num_blocks][num_kv_heads][block_size][head_dim]`` tensors.
``context_lens[s]`` counts the new token, which sits at logical position
``ctx - 1``; ``slot_mapping[s]`` is the flat pool slot of that position.
Block-table entries past a sequence's last block hold -1.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np
import torch

CHUNK = 1 << 24
DATA_SEED_BASE = 249000
META_SEED_BASE = 249100


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                 # "f32", "bf16" or "f16": dtype of q, pools and new K/V
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    partition_tokens: int      # 0 = library default, >0 = fixed split
    context_lens: np.ndarray   # int32 [S]
    block_tables: np.ndarray   # int32 [S][max_blocks_per_seq], -1 padded
    slot_mapping: np.ndarray   # int64 [S]
    q: torch.Tensor            # [S][H][D] (CPU)
    k_pool: torch.Tensor       # [NB][Hkv][BS][D] (CPU)
    v_pool: torch.Tensor
    new_key: torch.Tensor      # [S][Hkv][D] (CPU)
    new_value: torch.Tensor
    group_size: int = 1        # sequences per shared-prefix group (1 = none; uniform groups)
    prefix_len: int = 0        # shared-prefix tokens per group (uniform groups)
    group_starts: Optional[np.ndarray] = None  # int32 [G+1]: group i = seqs [gs[i], gs[i+1])
    group_prefix: Optional[np.ndarray] = None  # int32 [G]: tokens group i shares

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def kv_bytes_logical(self) -> int:
        """K+V bytes of all context tokens, counted per sequence."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * 2 * self.elem_bytes

    def kv_bytes_unique(self) -> int:
        """K+V bytes of distinct physical tokens (shared prefixes once)."""
        gs, gp = self.groups()
        ctx = self.context_lens.astype(np.int64)
        uniq = ctx.sum() - int(np.sum((np.diff(gs).astype(np.int64) - 1).clip(min=0) *
                                      gp.astype(np.int64)))
        return int(uniq) * self.num_kv_heads * self.head_dim * 2 * self.elem_bytes

    def groups(self) -> tuple[np.ndarray, np.ndarray]:
        """(group_starts int32 [G+1], prefix tokens int32 [G]) of the batch;
        a batch without sharing is one group per sequence with no prefix."""
        if self.group_starts is not None:
            return self.group_starts, self.group_prefix
        if self.group_size > 1:
            gs = np.arange(0, self.num_seqs + 1, self.group_size, dtype=np.int32)
            return gs, np.full(gs.size - 1, self.prefix_len, dtype=np.int32)
        return np.arange(self.num_seqs + 1, dtype=np.int32), np.zeros(self.num_seqs, np.int32)


def _normal_f32(ss: np.random.SeedSequence, n: int, threads: int = 0) -> np.ndarray:
    """n float32 N(0,1) draws, chunk i from grandchild stream i."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK
    kids = ss.spawn(nchunks)

    def fill(i: int) -> None:
        lo = i * CHUNK
        hi = min(n, lo + CHUNK)
        np.random.Generator(np.random.PCG64(kids[i])).standard_normal(
            hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        import os
        workers = threads or min(nchunks, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def _tensor(ss: np.random.SeedSequence, shape: Sequence[int], dtype: str) -> torch.Tensor:
    n = int(np.prod(shape)) if len(shape) else 1
    t = torch.from_numpy(_normal_f32(ss, n)).reshape(*shape)
    return t if dtype == "f32" else t.to(torch.bfloat16 if dtype == "bf16" else torch.float16)


def build(name: str, *, dtype: str, context_lens: Sequence[int], num_heads: int,
          num_kv_heads: int, head_dim: int, block_size: int, data_seed: int,
          meta_seed: int, placement: str = "shuffle", pool_blocks: Optional[int] = None,
          max_blocks_per_seq: Optional[int] = None, partition_tokens: int = 0,
          group_size: int = 1, prefix_len: int = 0, scale: Optional[float] = None,
          tail_fill: Optional[float] = None,
          groups: Optional[Sequence[tuple[int, int]]] = None) -> Workload:
    """Lay out a paged workload and fill it with seeded N(0,1) data.

    placement: "shuffle" (seeded permutation of the pool), "identity"
    (logical order = physical order), or "reverse".
    group_size/prefix_len: consecutive groups of ``group_size`` sequences
    share the physical blocks of their first ``prefix_len`` tokens
    (prefix_len must be a multiple of block_size).
    groups: ragged alternative, a list of (members, prefix_len): consecutive
    sequences form the groups in order (members summing to the batch).
    tail_fill: if given, every pool slot that no context position maps to is
    set to this value (e.g. NaN), to check that masked slots are ignored.
    """
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = int(ctx.size)
    BS = block_size
    if groups is None:
        if group_size > 1:
            assert S % group_size == 0
            groups = [(group_size, prefix_len)] * (S // group_size)
        else:
            groups = [(1, 0)] * S
    sizes = np.array([m for m, _ in groups], dtype=np.int64)
    gpref = np.array([p for _, p in groups], dtype=np.int64)
    assert int(sizes.sum()) == S and np.all(sizes >= 1) and np.all(gpref % BS == 0)
    gstart = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    seq_group = np.repeat(np.arange(len(groups)), sizes)
    for gi in range(len(groups)):
        assert np.all(ctx[gstart[gi]:gstart[gi + 1]] >= gpref[gi])
    nblk = (ctx + BS - 1) // BS
    gshared = np.where(sizes > 1, gpref // BS, 0)
    # unique logical blocks: per group the shared prefix once, then each
    # sequence's own blocks after the prefix
    owners = []  # (seq or -group-1 marker, logical block) for each unique block
    for s in range(S):
        gi = int(seq_group[s])
        if s == gstart[gi]:
            owners.extend(("p", gi, b) for b in range(int(gshared[gi])))
        owners.extend(("s", s, b) for b in range(int(gshared[gi]), int(nblk[s])))
    n_unique = len(owners)
    NB = int(pool_blocks) if pool_blocks is not None else n_unique
    assert NB >= n_unique
    rng = np.random.Generator(np.random.PCG64(meta_seed))
    if placement == "shuffle":
        perm = rng.permutation(NB)
    elif placement == "identity":
        perm = np.arange(NB)
    elif placement == "reverse":
        perm = np.arange(NB)[::-1].copy()
    else:
        raise ValueError(placement)
    MB = int(max_blocks_per_seq) if max_blocks_per_seq is not None else max(1, int(nblk.max()) if S else 1)
    assert S == 0 or MB >= int(nblk.max())
    bt = np.full((S, MB), -1, dtype=np.int32)
    prefix_phys = {}
    for i, (kind, a, b) in enumerate(owners):
        if kind == "p":
            prefix_phys[(a, b)] = int(perm[i])
        else:
            bt[a, b] = int(perm[i])
    for s in range(S):
        gi = int(seq_group[s])
        for b in range(int(gshared[gi])):
            bt[s, b] = prefix_phys[(gi, b)]
    slot = np.full(S, -1, dtype=np.int64)
    for s in range(S):
        if ctx[s] > 0:
            pos = int(ctx[s]) - 1
            slot[s] = int(bt[s, pos // BS]) * BS + pos % BS

    ss_q, ss_k, ss_v, ss_nk, ss_nv = np.random.SeedSequence(data_seed).spawn(5)
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    q = _tensor(ss_q, (S, H, D), dtype)
    k_pool = _tensor(ss_k, (NB, Hkv, BS, D), dtype)
    v_pool = _tensor(ss_v, (NB, Hkv, BS, D), dtype)
    nk = _tensor(ss_nk, (S, Hkv, D), dtype)
    nv = _tensor(ss_nv, (S, Hkv, D), dtype)
    if tail_fill is not None:
        used = np.zeros((NB, BS), dtype=bool)
        for s in range(S):
            for pos in range(int(ctx[s])):
                used[bt[s, pos // BS], pos % BS] = True
        mask = torch.from_numpy(~used)[:, None, :, None].expand(NB, Hkv, BS, D)
        k_pool[mask] = tail_fill
        v_pool[mask] = tail_fill
    return Workload(
        name=name, dtype=dtype, num_seqs=S, num_heads=H, num_kv_heads=Hkv, head_dim=D,
        block_size=BS, num_blocks=NB, max_blocks_per_seq=MB,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
        partition_tokens=partition_tokens, context_lens=ctx.astype(np.int32), block_tables=bt,
        slot_mapping=slot, q=q, k_pool=k_pool, v_pool=v_pool, new_key=nk, new_value=nv,
        group_size=group_size, prefix_len=prefix_len if group_size > 1 else 0,
        group_starts=gstart.astype(np.int32), group_prefix=np.where(sizes > 1, gpref, 0).astype(np.int32))


# The five decode workloads, by name. Sizes follow the PagedAttention decode
# setting: ragged context lengths, GQA head groups, a shared-prefix batch, and
# a long-context batch that needs the context split into partitions.
WORKLOADS = {
    "tiny_f32": dict(cid=1, desc="4 seqs, ctx {5,17,33,64}, 4/4 heads, D=64, BS=16, 32-block pool, fp32"),
    "mha_7b": dict(cid=2, desc="64 seqs, 32/32 heads, D=128, BS=16, ctx U[128,2048], bf16"),
    "gqa_8b": dict(cid=3, desc="128 seqs, 32/8 heads, D=128, BS=16, ctx U[512,8192], bf16"),
    "shared_prefix": dict(cid=4, desc="256 seqs = 32 groups x 8, 4096-token shared prefix + U[64,512] suffix, 32/8 heads, D=128, bf16"),
    "long_ctx": dict(cid=5, desc="8 seqs, ctx U[32768,131072], 64/8 heads, D=128, BS=16, partition 512, bf16"),
}


def lengths(name: str) -> np.ndarray:
    """Context lengths of a named workload (cheap: no data is drawn)."""
    cid = WORKLOADS[name]["cid"]
    rng = np.random.Generator(np.random.PCG64(META_SEED_BASE + cid))
    if name == "tiny_f32":
        return np.array([5, 17, 33, 64], dtype=np.int64)
    if name == "mha_7b":
        return rng.integers(128, 2048, size=64, endpoint=True)
    if name == "gqa_8b":
        return rng.integers(512, 8192, size=128, endpoint=True)
    if name == "shared_prefix":
        return 4096 + rng.integers(64, 512, size=256, endpoint=True)
    if name == "long_ctx":
        return rng.integers(32768, 131072, size=8, endpoint=True)
    raise KeyError(name)


def make(name: str, **overrides) -> Workload:
    """Build a named workload with its fixed seeds.

    ``overrides`` replace any keyword of ``build`` (dtype, head counts,
    head_dim, block_size, partition_tokens, ...); the block table is then
    sized from the workload's largest context for that block size.
    """
    cid = WORKLOADS[name]["cid"]
    ctx = lengths(name)
    # lengths() consumed the first draws of the meta stream; placement uses a
    # fresh stream derived from the same seed so it does not depend on that
    meta = META_SEED_BASE + cid + 1_000_000
    data = DATA_SEED_BASE + cid
    if name == "tiny_f32":
        kw = dict(dtype="f32", num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                  pool_blocks=32)
        max_tokens = 64
    elif name == "mha_7b":
        kw = dict(dtype="bf16", num_heads=32, num_kv_heads=32, head_dim=128, block_size=16)
        max_tokens = 2048
    elif name == "gqa_8b":
        kw = dict(dtype="bf16", num_heads=32, num_kv_heads=8, head_dim=128, block_size=16)
        max_tokens = 8192
    elif name == "shared_prefix":
        kw = dict(dtype="bf16", num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                  group_size=8, prefix_len=4096)
        max_tokens = 4096 + 512
    elif name == "long_ctx":
        kw = dict(dtype="bf16", num_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                  partition_tokens=512)
        max_tokens = 131072
    else:
        raise KeyError(name)
    kw.update(overrides)
    if "max_blocks_per_seq" not in overrides:
        kw["max_blocks_per_seq"] = -(-max_tokens // kw["block_size"])
    if name == "tiny_f32" and "pool_blocks" not in overrides and kw["block_size"] != 16:
        kw.pop("pool_blocks")  # the 32-block pool is sized for 16-token blocks
    return build(name, context_lens=ctx, data_seed=data, meta_seed=meta, **kw)


def subset(w: Workload, seqs: Sequence[int]) -> Workload:
    """The same pool with only the listed sequences in the batch."""
    idx = np.asarray(list(seqs), dtype=np.int64)
    return dataclasses.replace(
        w, num_seqs=int(idx.size), context_lens=w.context_lens[idx].copy(),
        block_tables=w.block_tables[idx].copy(), slot_mapping=w.slot_mapping[idx].copy(),
        q=w.q[torch.from_numpy(idx)].contiguous(), new_key=w.new_key[torch.from_numpy(idx)].contiguous(),
        new_value=w.new_value[torch.from_numpy(idx)].contiguous(), group_size=1, prefix_len=0,
        group_starts=None, group_prefix=None)
