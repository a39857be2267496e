"""Shared helpers of the GPU parity tests (not collected as tests)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_249_gb300 import pagedkv

# max-abs tolerances by input storage: fp32 1e-5 and bf16 2e-3 (fp32
# accumulation); fp16 inputs take the 16-bit input tolerance as well
TOL = {"f32": 1e-5, "bf16": 2e-3, "f16": 2e-3}


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (what storing an fp32 result as bf16 may add)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - 8).astype(np.int64))  # ulp = 2^(e-7); half = 2^(e-8)


def f16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half an fp16 ulp at |x| (what storing an fp32 result as fp16 may add;
    the subnormal spacing 2^-24 below 2^-14)."""
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - 11).astype(np.int64))  # ulp = 2^(e-10); half = 2^(e-11)


def oracle_after_write(w, seqs=None):
    """float64 oracle output of (a subset of) the batch after the cache write.

    The write is applied to copies of the host pools, so ``w`` is unchanged.
    """
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    assert oracle.reshape_and_cache(kp, vp, w.new_key, w.new_value, w.slot_mapping) == 0
    if seqs is None:
        return oracle.paged_decode(w.q, kp, vp, w.block_tables, w.context_lens, w.scale), kp, vp
    idx = np.asarray(seqs)
    ref = oracle.paged_decode(w.q[torch.from_numpy(idx)], kp, vp, w.block_tables[idx],
                              w.context_lens[idx], w.scale)
    return ref, kp, vp


def max_err(out: torch.Tensor, ref: np.ndarray) -> float:
    return float(np.abs(out.double().cpu().numpy() - ref).max()) if ref.size else 0.0


def assert_close(out: torch.Tensor, ref: np.ndarray, dtype: str, what: str = "") -> float:
    tol = TOL[dtype]
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if out.dtype in (torch.bfloat16, torch.float16):
        bound = tol + (bf16_half_ulp(ref) if out.dtype == torch.bfloat16 else f16_half_ulp(ref))
        bad = np.abs(got - ref) > bound
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond tol+half-ulp, max err " \
                              f"{np.abs(got - ref).max():.3g}"
        return float(np.abs(got - ref).max())
    err = max_err(out, ref)
    assert err <= tol, f"{what}: max abs error {err:.3g} > {tol}"
    return err


def run_decode(w, path=pagedkv.PATH_AUTO, partition_tokens=None, out_dtype=torch.float32,
               write=True):
    dw = pagedkv.DeviceWorkload(w, out_dtype=out_dtype, partition_tokens=partition_tokens)
    if write:
        dw.step(path=path)
    else:
        dw.decode(path=path)
    torch.cuda.synchronize()
    return dw
