"""float64 CPU oracle for paged decode attention and the cache write.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline arm are the only callers.  The CUDA library never
imports, links or calls anything here, and this package imports nothing from
the CUDA library.  The arithmetic lives in ``oracle.c`` (plain C, float64,
pthreads); this module compiles it with gcc and marshals arguments.

Definitions followed (see ``oracle.c`` for the full statement):
  * paged KV cache and block table -- Qualiteg, "About PagedAttention for LLM
    serving", the section on logical blocks, physical blocks and the block
    table that links them;
  * attention over the (non-contiguous) K and V -- vAttention, section 3.1
    "Requires re-writing the attention kernel" (standard softmax(q K^T scale) V,
    the formula the page names but does not print).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

F32, BF16, F16 = 0, 1, 2


def compile_source(src: str, out: str) -> str:
    """gcc a copy of oracle.c into a shared library (no fast-math, no FMA
    contraction, so x86 and Arm builds round alike)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-fno-fast-math", "-ffp-contract=off", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    lib = ctypes.CDLL(path)
    P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_paged_decode.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P, I, P, D, I]
    lib.oracle_paged_decode.restype = I
    lib.oracle_attention_contiguous.argtypes = [P, P, P, P, I, I, D]
    lib.oracle_attention_contiguous.restype = I
    lib.oracle_reshape_and_cache.argtypes = [P, P, I, I, I, I, I, P, P, P, I]
    lib.oracle_reshape_and_cache.restype = I
    return lib


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every call through another build of oracle.c (used
    by the tests that plant mistakes in a copy of the oracle)."""
    global _lib
    with _lock:
        saved, _lib = _lib, _open(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = _open(build())
            _lib = lib
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    raise TypeError(f"oracle supports float32, bfloat16 and float16 storage, got {t.dtype}")


def _cpu(t: torch.Tensor) -> torch.Tensor:
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous()


def paged_decode(query: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                 num_threads: int = 0) -> np.ndarray:
    """float64 [S][H][D] attention output of each sequence's single query.

    query [S][H][D]; pools [NB][Hkv][BS][D] (same dtype as query);
    block_tables int32 [S][max_blocks]; context_lens int32 [S].
    """
    lib = _load()
    q, kp, vp = _cpu(query), _cpu(k_pool), _cpu(v_pool)
    dt = _dtype_code(q)
    assert _dtype_code(kp) == dt and _dtype_code(vp) == dt
    S, H, D = q.shape
    NB, Hkv, BS, D2 = kp.shape
    assert D2 == D and tuple(vp.shape) == tuple(kp.shape)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32).reshape(S, -1)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32).reshape(S)
    out = np.zeros((S, H, D), dtype=np.float64)
    nt = num_threads or (os.cpu_count() or 1)
    rc = lib.oracle_paged_decode(out.ctypes.data, q.data_ptr(), kp.data_ptr(), vp.data_ptr(), dt,
                                 S, H, Hkv, D, BS, NB, bt.ctypes.data, bt.shape[1] if S else 0,
                                 cl.ctypes.data, float(scale), int(nt))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode rejected its input (status {rc})")
    return out


def attention_contiguous(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """float64 attention of one query row q[D] over contiguous K[ctx][D], V[ctx][D]."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64).reshape(-1, q.size)
    V = np.ascontiguousarray(V, dtype=np.float64).reshape(-1, q.size)
    assert K.shape == V.shape
    out = np.zeros(q.size, dtype=np.float64)
    rc = lib.oracle_attention_contiguous(out.ctypes.data, q.ctypes.data, K.ctypes.data,
                                         V.ctypes.data, K.shape[0], q.size, float(scale))
    if rc != 0:
        raise ValueError(f"oracle_attention_contiguous failed ({rc})")
    return out


def reshape_and_cache(k_pool: torch.Tensor, v_pool: torch.Tensor, key: torch.Tensor,
                      value: torch.Tensor, slot_mapping: np.ndarray) -> int:
    """In-place scatter of new K/V rows into CPU pools; returns #faulting slots."""
    lib = _load()
    assert k_pool.device.type == "cpu" and k_pool.is_contiguous() and v_pool.is_contiguous()
    dt = _dtype_code(k_pool)
    NB, Hkv, BS, D = k_pool.shape
    key, value = _cpu(key).to(k_pool.dtype), _cpu(value).to(k_pool.dtype)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert key.shape == (sm.size, Hkv, D) and value.shape == key.shape
    return lib.oracle_reshape_and_cache(k_pool.data_ptr(), v_pool.data_ptr(), dt, NB, BS, Hkv, D,
                                        key.data_ptr(), value.data_ptr(), sm.ctypes.data, sm.size)
