"""The host block manager (C++ behind the C ABI), on the CPU.

A host mirror of the pool records which token every slot holds.  After any
sequence of add / fork / append / free operations, gathering each live
sequence through its block table must give back exactly its token history,
reference counts must equal the number of sequences holding each block, and
free blocks must be exactly the unreferenced ones.
"""
import numpy as np
import pytest

from paged_kv_cache_249_gb300 import build as pkv_build
from paged_kv_cache_249_gb300 import pagedkv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    pagedkv.load()


class Mirror:
    def __init__(self, nb, bs):
        self.nb, self.bs = nb, bs
        self.pool = np.full(nb * bs, -1, dtype=np.int64)
        self.hist = {}
        self.next_tok = 0

    def tok(self):
        self.next_tok += 1
        return self.next_tok

    def apply_copies(self, bm):
        src, dst = bm.take_copies()
        for s, d in zip(src, dst):
            self.pool[d * self.bs:(d + 1) * self.bs] = self.pool[s * self.bs:(s + 1) * self.bs]

    def check(self, bm):
        ids = sorted(self.hist)
        if ids:
            mb = max(1, max(-(-len(self.hist[i]) // self.bs) for i in ids))
            bt, cl = bm.block_tables(ids, mb)
            refs = np.zeros(self.nb, dtype=np.int64)
            for row, i, n in zip(bt, ids, cl):
                assert n == len(self.hist[i]) == bm.context_len(i)
                got = [self.pool[row[p // self.bs] * self.bs + p % self.bs] for p in range(n)]
                assert got == self.hist[i], f"sequence {i}"
                for b in row[row >= 0]:
                    refs[b] += 1
        else:
            refs = np.zeros(self.nb, dtype=np.int64)
        for b in range(self.nb):
            assert bm.refcount(b) == refs[b]
        assert bm.free_blocks == int((refs == 0).sum())


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_every_sequence_intact(seed):
    rng = np.random.default_rng(seed)
    nb, bs = 48, int(rng.choice([2, 4, 16]))
    bm = pagedkv.BlockManager(nb, bs)
    m = Mirror(nb, bs)
    next_id = 0
    for step in range(400):
        op = rng.choice(["add", "fork", "append", "append", "append", "free"])
        live = sorted(m.hist)
        try:
            if op == "add" or not live:
                n = int(rng.integers(0, 3 * bs))
                slots = bm.add_sequence(next_id, n)
                toks = [m.tok() for _ in range(n)]
                m.pool[slots] = toks
                m.hist[next_id] = toks
                next_id += 1
            elif op == "fork":
                p = int(rng.choice(live))
                bm.fork(p, next_id)
                m.hist[next_id] = list(m.hist[p])
                next_id += 1
            elif op == "append":
                i = int(rng.choice(live))
                slot = bm.append_token(i)
                m.apply_copies(bm)          # copy-on-write before the write
                t = m.tok()
                m.pool[slot] = t
                m.hist[i].append(t)
            else:
                i = int(rng.choice(live))
                bm.free_sequence(i)
                del m.hist[i]
        except pagedkv.PagedKVError as e:
            assert e.status == pagedkv.ERR_OUT_OF_BLOCKS
        m.check(bm)


def test_out_of_blocks_leaves_state_unchanged():
    bm = pagedkv.BlockManager(3, 4)
    bm.add_sequence(0, 12)  # all three blocks
    assert bm.free_blocks == 0
    with pytest.raises(pagedkv.PagedKVError) as e:
        bm.add_sequence(1, 1)
    assert e.value.status == pagedkv.ERR_OUT_OF_BLOCKS
    with pytest.raises(pagedkv.PagedKVError):
        bm.append_token(0)  # needs a fourth block
    assert bm.context_len(0) == 12 and bm.context_len(1) == -1
    bm.free_sequence(0)
    assert bm.free_blocks == 3


def test_fork_shares_then_copies_on_write():
    bm = pagedkv.BlockManager(8, 4)
    bm.add_sequence(7, 6)            # blocks 0 (full) and 1 (2 of 4 rows)
    bm.fork(7, 8)
    assert bm.refcount(0) == 2 and bm.refcount(1) == 2
    slot = bm.append_token(8)        # writes into the shared partial block
    src, dst = bm.take_copies()
    assert list(src) == [1] and list(dst) == [2] and slot == 2 * 4 + 2
    assert bm.refcount(1) == 1 and bm.refcount(2) == 1 and bm.refcount(0) == 2
    assert bm.append_token(7) == 1 * 4 + 2  # the parent keeps its own block, no copy
    assert bm.take_copies()[0].size == 0
    bt, cl = bm.block_tables([7, 8], 3)
    assert bt.tolist() == [[0, 1, -1], [0, 2, -1]] and cl.tolist() == [7, 7]


def test_invalid_arguments():
    lib = pagedkv.load()
    import ctypes
    h = ctypes.c_void_p()
    assert lib.pkv_bm_create(0, 16, ctypes.byref(h)) == pagedkv.ERR_INVALID_ARG
    assert lib.pkv_bm_free_blocks(None) == -1
    bm = pagedkv.BlockManager(4, 16)
    bm.add_sequence(1, 3)
    for call in (lambda: bm.add_sequence(1, 2), lambda: bm.fork(5, 6), lambda: bm.fork(1, 1),
                 lambda: bm.append_token(9), lambda: bm.free_sequence(9),
                 lambda: bm.block_tables([9], 4), lambda: bm.add_sequence(2, -1)):
        with pytest.raises(pagedkv.PagedKVError) as e:
            call()
        assert e.value.status == pagedkv.ERR_INVALID_ARG
    with pytest.raises(pagedkv.PagedKVError):
        bm.block_tables([1], 0)


def test_shared_prefix_of_forked_sequences():
    """Forked sequences share their parent's full blocks; a partly filled
    last block is not counted, and copy-on-write does not change the count
    of full shared blocks."""
    bm = pagedkv.BlockManager(64, 16)
    bm.add_sequence(0, 70)  # 4 full blocks + 6 tokens
    bm.fork(0, 1)
    bm.fork(0, 2)
    bm.add_sequence(3, 20)
    assert bm.shared_prefix([0, 1, 2, 3], [0, 3, 4]).tolist() == [64, 0]
    bm.append_token(1)  # private copy of the partial last block
    assert bm.shared_prefix([0, 1, 2, 3], [0, 3, 4]).tolist() == [64, 0]
    # sequences that share nothing, listed as one group
    assert bm.shared_prefix([0, 3], [0, 2]).tolist() == [0]
    # a group of one shares nothing
    assert bm.shared_prefix([0, 1], [0, 1, 2]).tolist() == [0, 0]
    # fill the shared partial block region in every member: still 4 blocks
    # until the members' fifth blocks differ (after copy-on-write they do)
    for _ in range(10):
        for s in (0, 1, 2):
            bm.append_token(s)
    assert bm.shared_prefix([0, 1, 2], [0, 3]).tolist() == [64]
    with pytest.raises(pagedkv.PagedKVError):
        bm.shared_prefix([0, 99], [0, 2])  # unknown sequence
    with pytest.raises(pagedkv.PagedKVError):
        bm.shared_prefix([0, 1], [0, 1])  # groups do not cover the list
