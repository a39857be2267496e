"""Thin ctypes binding over libpagedkv.so (the C ABI of include/pagedkv.h).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or was built
for another machine, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

# pkv_status
(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_DEVICE_FAULT,
 ERR_OUT_OF_BLOCKS) = range(7)
# pkv_dtype
F32, BF16, F16 = 0, 1, 2
# device fault bits
FAULT_BLOCK_ID, FAULT_SLOT, FAULT_CONTEXT, FAULT_TIMEOUT, FAULT_PREFIX = 1, 2, 4, 8, 16
# decode paths
PATH_AUTO, PATH_FMA, PATH_MMA = 0, 1, 2

EXPORTS = ["pkv_pool_bytes", "pkv_block_pool_init", "pkv_block_table_upload",
           "pkv_reshape_and_cache", "pkv_decode_workspace_bytes", "pkv_paged_attention_decode",
           "pkv_get_device_error", "pkv_status_string", "pkv_version",
           "pkv_paged_attention_decode_static", "pkv_last_cuda_error", "pkv_copy_blocks",
           "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_free_blocks", "pkv_bm_refcount",
           "pkv_bm_add_sequence", "pkv_bm_fork", "pkv_bm_append_token", "pkv_bm_free_sequence",
           "pkv_bm_context_len", "pkv_bm_pending_copies", "pkv_bm_take_copies",
           "pkv_bm_block_tables", "pkv_bm_shared_prefix", "pkv_contiguous_cache_init",
           "pkv_contiguous_attention_decode", "pkv_shared_prefix_workspace_bytes",
           "pkv_paged_attention_decode_shared_prefix", "pkv_shared_prefix_plan",
           "pkv_paged_attention_decode_shared_prefix_run", "pkv_check_bounded_wait"]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        if status == ERR_CUDA and _lib is not None:
            msg += ": " + _lib.pkv_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")


class pkv_pool(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("num_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("device", ctypes.c_int),
                ("layout", ctypes.c_int), ("num_seqs", ctypes.c_int), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("dev_error", ctypes.c_void_p), ("tma", ctypes.c_uint64 * 32)]


_lib = None


def load(path: Optional[str] = None):
    """Load libpagedkv.so and declare its signatures (raises if absent)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with paged_kv_cache_249_gb300.build.build()")
    lib = ctypes.CDLL(p)
    I, P, Z, F = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    L = ctypes.c_int64
    PP = ctypes.POINTER(pkv_pool)
    sig = {
        "pkv_pool_bytes": (Z, [I, I, I, I, I]),
        "pkv_block_pool_init": (I, [PP, I, I, I, I, I, P, P, P, I, P]),
        "pkv_block_table_upload": (I, [P, P, I, I, I, P]),
        "pkv_reshape_and_cache": (I, [PP, P, P, P, I, P]),
        "pkv_decode_workspace_bytes": (Z, [I, I, I, I, I]),
        "pkv_paged_attention_decode": (I, [PP, P, I, P, I, I, I, P, I, P, I, F, I, P, Z, I, P]),
        "pkv_get_device_error": (I, [PP, P, ctypes.POINTER(ctypes.c_uint32)]),
        "pkv_check_bounded_wait": (I, [PP, ctypes.c_longlong, P]),
        "pkv_paged_attention_decode_static": (I, [PP, P, I, P, I, I, I, P, I, P, I, F, I, I, P]),
        "pkv_copy_blocks": (I, [PP, P, P, I, P]),
        "pkv_contiguous_cache_init": (I, [PP, I, I, I, I, I, P, P, P, I, P]),
        "pkv_contiguous_attention_decode": (I, [PP, P, I, P, I, I, I, P, I, F, I, P, Z, I, P]),
        "pkv_shared_prefix_workspace_bytes": (Z, [I, I, I, I, I, I]),
        "pkv_paged_attention_decode_shared_prefix": (I, [PP, P, I, P, I, I, I, P, I, P, I, F, P, P,
                                                         I, I, I, P, Z, P]),
        "pkv_shared_prefix_plan": (I, [PP, I, I, I, I, P, I, P, P, I, I, I, P, Z, P]),
        "pkv_paged_attention_decode_shared_prefix_run": (I, [PP, P, I, P, I, I, I, P, I, I, F, I, I,
                                                             P, Z, P]),
        "pkv_bm_create": (I, [I, I, ctypes.POINTER(P)]),
        "pkv_bm_destroy": (None, [P]),
        "pkv_bm_free_blocks": (I, [P]),
        "pkv_bm_refcount": (I, [P, ctypes.c_int32]),
        "pkv_bm_add_sequence": (I, [P, L, L, P]),
        "pkv_bm_fork": (I, [P, L, L]),
        "pkv_bm_append_token": (I, [P, L, ctypes.POINTER(L)]),
        "pkv_bm_free_sequence": (I, [P, L]),
        "pkv_bm_context_len": (L, [P, L]),
        "pkv_bm_pending_copies": (I, [P]),
        "pkv_bm_take_copies": (I, [P, P, P, I]),
        "pkv_bm_block_tables": (I, [P, P, I, I, P, P]),
        "pkv_bm_shared_prefix": (I, [P, P, I, P, I, P]),
        "pkv_status_string": (ctypes.c_char_p, [I]),
        "pkv_last_cuda_error": (ctypes.c_char_p, []),
        "pkv_version": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise PagedKVError(status, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float16:
        return F16
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def pool_bytes(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
               dtype: torch.dtype) -> int:
    return load().pkv_pool_bytes(num_blocks, block_size, num_kv_heads, head_dim, _dtype_code(dtype))


class BlockPool:
    """A caller-owned K/V block pool described to the library."""

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 dev_error: Optional[torch.Tensor] = None, zero_fill: bool = False,
                 stream: Optional[torch.cuda.Stream] = None):
        assert k_pool.shape == v_pool.shape and k_pool.dtype == v_pool.dtype
        assert k_pool.is_contiguous() and v_pool.is_contiguous()
        NB, Hkv, BS, D = k_pool.shape
        self.k_pool, self.v_pool, self.dev_error = k_pool, v_pool, dev_error
        self.desc = pkv_pool()
        _check(load().pkv_block_pool_init(ctypes.byref(self.desc), NB, BS, Hkv, D,
                                          _dtype_code(k_pool.dtype), k_pool.data_ptr(),
                                          v_pool.data_ptr(), _ptr(dev_error), int(zero_fill),
                                          _stream(stream)), "pkv_block_pool_init")

    @property
    def num_blocks(self) -> int:
        return self.desc.num_blocks

    @property
    def block_size(self) -> int:
        return self.desc.block_size

    @property
    def num_kv_heads(self) -> int:
        return self.desc.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.desc.head_dim


def block_pool_init(k_pool, v_pool, dev_error=None, zero_fill=False, stream=None) -> BlockPool:
    return BlockPool(k_pool, v_pool, dev_error, zero_fill, stream)


def block_table_upload(dev_block_tables: torch.Tensor, host_block_tables: torch.Tensor,
                       num_blocks: int = 0, stream=None) -> None:
    """Asynchronous H2D copy of an int32 [S][max_blocks] table (host tensor
    should be pinned and must stay alive until the copy has run)."""
    assert host_block_tables.dtype == torch.int32 and host_block_tables.is_contiguous()
    assert dev_block_tables.dtype == torch.int32 and dev_block_tables.is_contiguous()
    S, MB = host_block_tables.shape
    assert tuple(dev_block_tables.shape) == (S, MB)
    _check(load().pkv_block_table_upload(dev_block_tables.data_ptr(), host_block_tables.data_ptr(),
                                         S, MB, num_blocks, _stream(stream)),
           "pkv_block_table_upload")


def reshape_and_cache(pool: BlockPool, key: torch.Tensor, value: torch.Tensor,
                      slot_mapping: torch.Tensor, stream=None) -> None:
    assert slot_mapping.dtype == torch.int64
    _check(load().pkv_reshape_and_cache(ctypes.byref(pool.desc), key.data_ptr(), value.data_ptr(),
                                        slot_mapping.data_ptr(), slot_mapping.numel(),
                                        _stream(stream)), "pkv_reshape_and_cache")


def decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                           partition_tokens: int = 0) -> int:
    return load().pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                             partition_tokens)


def paged_attention_decode(pool: BlockPool, out: torch.Tensor, query: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           max_context_len: int, scale: float, num_kv_heads: Optional[int] = None,
                           partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                           path: int = PATH_AUTO, stream=None) -> None:
    S, H, _ = query.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_paged_attention_decode(
        ctypes.byref(pool.desc), out.data_ptr(), _dtype_code(out.dtype), query.data_ptr(), S, H,
        num_kv_heads if num_kv_heads is not None else pool.num_kv_heads, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), int(max_context_len), float(scale),
        int(partition_tokens), _ptr(workspace), ws_bytes, int(path), _stream(stream)),
        "pkv_paged_attention_decode")


STATIC_SCRATCH_BYTES = 64 << 20


def paged_attention_decode_static(pool: BlockPool, out: torch.Tensor, query: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  max_context_len: int, scale: float,
                                  num_kv_heads: Optional[int] = None, partition_tokens: int = 0,
                                  path: int = PATH_AUTO, stream=None) -> None:
    """pkv_paged_attention_decode_static: the same decode with its split-K
    partials in the library's fixed device array (no workspace argument, no
    allocation).  For callers that cannot allocate device memory; calls that
    overlap on the GPU share that array and race."""
    S, H, _ = query.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    _check(load().pkv_paged_attention_decode_static(
        ctypes.byref(pool.desc), out.data_ptr(), _dtype_code(out.dtype), query.data_ptr(), S, H,
        num_kv_heads if num_kv_heads is not None else pool.num_kv_heads, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), int(max_context_len), float(scale),
        int(partition_tokens), int(path), _stream(stream)), "pkv_paged_attention_decode_static")


def shared_prefix_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int,
                                  max_context_len: int, max_prefix_len: int,
                                  partition_tokens: int = 0) -> int:
    return load().pkv_shared_prefix_workspace_bytes(num_seqs, num_heads, head_dim,
                                                    max_context_len, max_prefix_len,
                                                    partition_tokens)


def paged_attention_decode_shared_prefix(pool: BlockPool, out: torch.Tensor, query: torch.Tensor,
                                         block_tables: torch.Tensor, context_lens: torch.Tensor,
                                         max_context_len: int, scale: float,
                                         group_starts: torch.Tensor, prefix_lens: torch.Tensor,
                                         max_prefix_len: int, workspace: torch.Tensor,
                                         num_kv_heads: Optional[int] = None,
                                         partition_tokens: int = 0, stream=None) -> None:
    """pkv_paged_attention_decode_shared_prefix: decode for a batch whose
    groups of sequences (group_starts, int32 [G+1]) share the blocks of a
    prompt prefix (prefix_lens, int32 [G], tokens)."""
    S, H, _ = query.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert group_starts.dtype == torch.int32 and prefix_lens.dtype == torch.int32
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_attention_decode_shared_prefix(
        ctypes.byref(pool.desc), out.data_ptr(), _dtype_code(out.dtype), query.data_ptr(), S, H,
        num_kv_heads if num_kv_heads is not None else pool.num_kv_heads, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), int(max_context_len), float(scale),
        group_starts.data_ptr(), prefix_lens.data_ptr(), prefix_lens.numel(),
        int(max_prefix_len), int(partition_tokens), workspace.data_ptr(), ws_bytes,
        _stream(stream)), "pkv_paged_attention_decode_shared_prefix")


def shared_prefix_plan(pool: BlockPool, num_heads: int, context_lens: torch.Tensor,
                       max_context_len: int, group_starts: torch.Tensor,
                       prefix_lens: torch.Tensor, max_prefix_len: int, workspace: torch.Tensor,
                       max_blocks_per_seq: int, num_kv_heads: Optional[int] = None,
                       partition_tokens: int = 0, stream=None) -> None:
    """pkv_shared_prefix_plan: the work list of a shared-prefix decode, reusable
    by every layer of the step."""
    _check(load().pkv_shared_prefix_plan(
        ctypes.byref(pool.desc), context_lens.numel(), num_heads,
        num_kv_heads if num_kv_heads is not None else pool.num_kv_heads, int(max_blocks_per_seq),
        context_lens.data_ptr(), int(max_context_len), group_starts.data_ptr(),
        prefix_lens.data_ptr(), prefix_lens.numel(), int(max_prefix_len), int(partition_tokens),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "pkv_shared_prefix_plan")


def paged_attention_decode_shared_prefix_run(pool: BlockPool, out: torch.Tensor,
                                             query: torch.Tensor, block_tables: torch.Tensor,
                                             max_context_len: int, scale: float,
                                             max_prefix_len: int, workspace: torch.Tensor,
                                             num_kv_heads: Optional[int] = None,
                                             partition_tokens: int = 0, stream=None) -> None:
    """pkv_paged_attention_decode_shared_prefix_run: decode from the plan in
    `workspace`."""
    S, H, _ = query.shape
    _check(load().pkv_paged_attention_decode_shared_prefix_run(
        ctypes.byref(pool.desc), out.data_ptr(), _dtype_code(out.dtype), query.data_ptr(), S, H,
        num_kv_heads if num_kv_heads is not None else pool.num_kv_heads, block_tables.data_ptr(),
        block_tables.shape[1], int(max_context_len), float(scale), int(max_prefix_len),
        int(partition_tokens), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(stream)), "pkv_paged_attention_decode_shared_prefix_run")


class ContiguousCache:
    """A conventional [S][Hkv][capacity][D] K/V cache (the layout a paged
    pool replaces), described to the library for the paging-overhead
    comparison."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 dev_error: Optional[torch.Tensor] = None, stream=None):
        assert k_cache.shape == v_cache.shape and k_cache.is_contiguous() and v_cache.is_contiguous()
        S, Hkv, cap, D = k_cache.shape
        self.k_cache, self.v_cache, self.dev_error = k_cache, v_cache, dev_error
        self.desc = pkv_pool()
        _check(load().pkv_contiguous_cache_init(ctypes.byref(self.desc), S, cap, Hkv, D,
                                                _dtype_code(k_cache.dtype), k_cache.data_ptr(),
                                                v_cache.data_ptr(), _ptr(dev_error), 0,
                                                _stream(stream)), "pkv_contiguous_cache_init")
        self.num_kv_heads = Hkv

    @staticmethod
    def from_paged(w, capacity: Optional[int] = None, device="cuda", k_pool=None,
                   v_pool=None) -> "ContiguousCache":
        """Gather a paged Workload's tokens (logical order) into a contiguous
        cache, from its host pools or from the given (device) pools."""
        BS = w.block_size
        cap = capacity or max(BS, -(-w.max_context_len // BS) * BS)
        S, Hkv, D = w.num_seqs, w.num_kv_heads, w.head_dim
        k = torch.zeros(S, Hkv, cap, D, dtype=w.torch_dtype, device=device)
        v = torch.zeros_like(k)
        kp = (k_pool if k_pool is not None else w.k_pool).to(device)
        vp = (v_pool if v_pool is not None else w.v_pool).to(device)
        for s in range(S):
            n = int(w.context_lens[s])
            nb = -(-n // BS)
            if nb == 0:
                continue
            blocks = torch.from_numpy(w.block_tables[s, :nb].astype(np.int64)).to(device)
            # [nb][Hkv][BS][D] -> [Hkv][nb*BS][D]
            k[s, :, :nb * BS] = kp[blocks].permute(1, 0, 2, 3).reshape(Hkv, nb * BS, D)
            v[s, :, :nb * BS] = vp[blocks].permute(1, 0, 2, 3).reshape(Hkv, nb * BS, D)
        return ContiguousCache(k, v)


def contiguous_attention_decode(cache: ContiguousCache, out: torch.Tensor, query: torch.Tensor,
                                context_lens: torch.Tensor, max_context_len: int, scale: float,
                                partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                                path: int = PATH_AUTO, stream=None) -> None:
    S, H, _ = query.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pkv_contiguous_attention_decode(
        ctypes.byref(cache.desc), out.data_ptr(), _dtype_code(out.dtype), query.data_ptr(), S, H,
        cache.num_kv_heads, context_lens.data_ptr(), int(max_context_len), float(scale),
        int(partition_tokens), _ptr(workspace), ws_bytes, int(path), _stream(stream)),
        "pkv_contiguous_attention_decode")


def copy_blocks(pool: BlockPool, src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """Device copy of whole blocks src[i] -> dst[i] (int32 device tensors)."""
    assert src.dtype == torch.int32 and dst.dtype == torch.int32 and src.numel() == dst.numel()
    _check(load().pkv_copy_blocks(ctypes.byref(pool.desc), src.data_ptr(), dst.data_ptr(),
                                  src.numel(), _stream(stream)), "pkv_copy_blocks")


class BlockManager:
    """Host block manager of a pool (C++ behind the C ABI; host memory only)."""

    def __init__(self, num_blocks: int, block_size: int):
        self.lib = load()
        self.block_size = block_size
        h = ctypes.c_void_p()
        _check(self.lib.pkv_bm_create(num_blocks, block_size, ctypes.byref(h)), "pkv_bm_create")
        self.h = h

    def __del__(self):
        if getattr(self, "h", None) and self.h.value:
            self.lib.pkv_bm_destroy(self.h)
            self.h = None

    @property
    def free_blocks(self) -> int:
        return self.lib.pkv_bm_free_blocks(self.h)

    def refcount(self, block: int) -> int:
        return self.lib.pkv_bm_refcount(self.h, block)

    def add_sequence(self, seq_id: int, num_tokens: int) -> np.ndarray:
        slots = np.empty(max(num_tokens, 1), dtype=np.int64)
        _check(self.lib.pkv_bm_add_sequence(self.h, seq_id, num_tokens, slots.ctypes.data),
               "pkv_bm_add_sequence")
        return slots[:num_tokens]

    def fork(self, parent: int, child: int) -> None:
        _check(self.lib.pkv_bm_fork(self.h, parent, child), "pkv_bm_fork")

    def append_token(self, seq_id: int) -> int:
        slot = ctypes.c_int64(-1)
        _check(self.lib.pkv_bm_append_token(self.h, seq_id, ctypes.byref(slot)),
               "pkv_bm_append_token")
        return slot.value

    def free_sequence(self, seq_id: int) -> None:
        _check(self.lib.pkv_bm_free_sequence(self.h, seq_id), "pkv_bm_free_sequence")

    def context_len(self, seq_id: int) -> int:
        return self.lib.pkv_bm_context_len(self.h, seq_id)

    def take_copies(self):
        n = self.lib.pkv_bm_pending_copies(self.h)
        src = np.empty(max(n, 1), dtype=np.int32)
        dst = np.empty(max(n, 1), dtype=np.int32)
        got = self.lib.pkv_bm_take_copies(self.h, src.ctypes.data, dst.ctypes.data, n)
        return src[:got], dst[:got]

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        bt = np.empty((ids.size, max_blocks_per_seq), dtype=np.int32)
        cl = np.empty(ids.size, dtype=np.int32)
        _check(self.lib.pkv_bm_block_tables(self.h, ids.ctypes.data, ids.size, max_blocks_per_seq,
                                            bt.ctypes.data, cl.ctypes.data),
               "pkv_bm_block_tables")
        return bt, cl

    def shared_prefix(self, seq_ids, group_starts) -> np.ndarray:
        """Tokens of the leading full blocks each group's members share."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        gs = np.ascontiguousarray(group_starts, dtype=np.int32)
        out = np.zeros(max(gs.size - 1, 1), dtype=np.int32)
        _check(self.lib.pkv_bm_shared_prefix(self.h, ids.ctypes.data, ids.size, gs.ctypes.data,
                                             gs.size - 1, out.ctypes.data),
               "pkv_bm_shared_prefix")
        return out[:gs.size - 1]


def get_device_error(pool: BlockPool, stream=None) -> int:
    """Synchronise, return and clear the pool's device fault bits."""
    bits = ctypes.c_uint32(0)
    st = load().pkv_get_device_error(ctypes.byref(pool.desc), _stream(stream), ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE_FAULT):
        _check(st, "pkv_get_device_error")
    return int(bits.value)


def check_bounded_wait(pool: BlockPool, limit_ns: int, stream=None) -> None:
    """pkv_check_bounded_wait: run the kernels' bounded pipeline wait on a
    barrier nothing arrives at, with limit_ns as the bound (it sets
    FAULT_TIMEOUT in the pool's error word)."""
    _check(load().pkv_check_bounded_wait(ctypes.byref(pool.desc), int(limit_ns), _stream(stream)),
           "pkv_check_bounded_wait")


def alloc_workspace(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                    partition_tokens: int = 0, device=None) -> Optional[torch.Tensor]:
    """A torch-owned workspace buffer of the size the library asks for."""
    n = decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_tokens)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


class DeviceWorkload:
    """A Workload's tensors resident on the GPU, with its pool described."""

    def __init__(self, w, device="cuda", out_dtype: Optional[torch.dtype] = None,
                 partition_tokens: Optional[int] = None):
        self.w = w
        self.q = w.q.to(device)
        self.k_pool = w.k_pool.to(device)
        self.v_pool = w.v_pool.to(device)
        self.new_key = w.new_key.to(device)
        self.new_value = w.new_value.to(device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.context_lens = torch.from_numpy(w.context_lens).to(device)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(device)
        self.device = device
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=device)
        self.pool = BlockPool(self.k_pool, self.v_pool, self.dev_error)
        self.out = torch.empty(w.num_seqs, w.num_heads, w.head_dim,
                               dtype=out_dtype or torch.float32, device=device)
        self.partition_tokens = w.partition_tokens if partition_tokens is None else partition_tokens
        self.max_context_len = max(1, w.max_context_len)
        self.workspace = alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, self.max_context_len,
                                         self.partition_tokens, device)

    def step(self, path: int = PATH_AUTO, stream=None) -> None:
        """One decode step: cache write of the new tokens, then attention."""
        reshape_and_cache(self.pool, self.new_key, self.new_value, self.slot_mapping, stream)
        self.decode(path=path, stream=stream)

    def decode(self, path: int = PATH_AUTO, stream=None) -> None:
        paged_attention_decode(self.pool, self.out, self.q, self.block_tables, self.context_lens,
                               self.max_context_len, self.w.scale, self.w.num_kv_heads,
                               self.partition_tokens, self.workspace, path, stream)

    def shared_prefix_setup(self, partition_tokens: int = 0, group_starts=None,
                            prefix_lens=None, max_prefix_len: Optional[int] = None) -> None:
        """Upload the batch's group description (or the one given) and size the
        shared-prefix workspace."""
        gs, gp = self.w.groups()
        gs = gs if group_starts is None else np.asarray(group_starts, dtype=np.int32)
        gp = gp if prefix_lens is None else np.asarray(prefix_lens, dtype=np.int32)
        self.group_starts = torch.from_numpy(np.ascontiguousarray(gs)).to(self.device)
        self.prefix_lens = torch.from_numpy(np.ascontiguousarray(gp)).to(self.device)
        self.max_prefix_len = int(max_prefix_len if max_prefix_len is not None else
                                  (max(0, int(gp.max())) if gp.size else 0))
        self.sp_partition = partition_tokens
        n = shared_prefix_workspace_bytes(self.w.num_seqs, self.w.num_heads, self.w.head_dim,
                                          self.max_context_len, self.max_prefix_len,
                                          partition_tokens)
        self.sp_workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)

    def decode_shared_prefix(self, stream=None) -> None:
        if not hasattr(self, "sp_workspace"):
            self.shared_prefix_setup()
        paged_attention_decode_shared_prefix(
            self.pool, self.out, self.q, self.block_tables, self.context_lens,
            self.max_context_len, self.w.scale, self.group_starts, self.prefix_lens,
            self.max_prefix_len, self.sp_workspace, self.w.num_kv_heads, self.sp_partition, stream)

    def shared_prefix_plan(self, stream=None) -> None:
        if not hasattr(self, "sp_workspace"):
            self.shared_prefix_setup()
        shared_prefix_plan(self.pool, self.w.num_heads, self.context_lens, self.max_context_len,
                           self.group_starts, self.prefix_lens, self.max_prefix_len,
                           self.sp_workspace, self.block_tables.shape[1], self.w.num_kv_heads,
                           self.sp_partition, stream)

    def decode_shared_prefix_run(self, stream=None) -> None:
        paged_attention_decode_shared_prefix_run(
            self.pool, self.out, self.q, self.block_tables, self.max_context_len, self.w.scale,
            self.max_prefix_len, self.sp_workspace, self.w.num_kv_heads, self.sp_partition, stream)
