"""Full-size decode workloads, in the launch configuration the benchmark
times (bf16 output, automatic or workload-given partitioning, automatic
compute path), compared with the float64 oracle on every sequence and every
element; the shared-prefix batch also with 256- and 64-wide heads (their
items carry 16 query rows) and with fp32 pools (TF32 tiles), which take the
plan's longer automatic prefix parts (1024 and 2048 tokens), the GQA batch
with fp16 pools and the MHA batch in 64-token blocks.

The oracle computes each sequence's result through its own block table
(Qualiteg, "About PagedAttention for LLM serving", the section on logical
blocks, physical blocks and the block table that links them); the cache write
before the decode is compared bit for bit over the whole pool, so a slot
written in the wrong place, or a stray write anywhere else, fails.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu

FULL = ["mha_7b", "gqa_8b", "shared_prefix", "long_ctx", "shared_prefix/head_dim=256",
        "shared_prefix/head_dim=64", "shared_prefix/dtype=f32", "gqa_8b/dtype=f16",
        "mha_7b/block_size=64"]


def _make(param):
    """A workload by name, with an optional shape override after a slash."""
    name, _, over = param.partition("/")
    kw = {}
    if over:
        k, v = over.split("=")
        kw[k] = v if k == "dtype" else int(v)
    return workload.make(name, **kw)


def _tol(w):
    return {"f16": "f16", "f32": "f32"}.get(w.dtype, "bf16")


def _bits(t: torch.Tensor) -> torch.Tensor:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.fixture(scope="module", params=FULL)
def full(request):
    """A full-size workload with the oracle's pools after the cache write and
    its float64 output for the whole batch."""
    w = _make(request.param)
    ref, kp, vp = oracle_after_write(w)
    yield request.param, w, ref, kp, vp


def test_fullsize_cache_write_bit_exact_pool_wide(full):
    name, w, _, kp, vp = full
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    assert torch.equal(_bits(dw.k_pool), _bits(kp)), f"{name}: K pool differs after the write"
    assert torch.equal(_bits(dw.v_pool), _bits(vp)), f"{name}: V pool differs after the write"


def test_fullsize_plain_decode_whole_batch(full):
    name, w, ref, _, _ = full
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    dw.step()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    assert_close(dw.out, ref, _tol(w), f"{name} bf16 output, all {w.num_seqs} sequences")
    # the same launch with fp32 output, graded at the tolerance alone
    dw32 = pagedkv.DeviceWorkload(w, out_dtype=torch.float32)
    dw32.step()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw32.pool) == 0
    assert_close(dw32.out, ref, _tol(w), f"{name} fp32 output, all {w.num_seqs} sequences")
    # the bf16 output is the fp32 output rounded once
    assert torch.equal(_bits(dw32.out.to(torch.bfloat16)), _bits(dw.out))


def test_fullsize_shared_prefix_decode_whole_batch(full):
    """The shared-prefix entry point on every full-size workload: batches
    without groups are one sequence per group (no sharing); the
    shared-prefix batch reads each group's 4096-token prefix once per kv head."""
    name, w, ref, _, _ = full
    for out_dtype in (torch.float32, torch.bfloat16):
        dw = pagedkv.DeviceWorkload(w, out_dtype=out_dtype)
        pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
        dw.shared_prefix_setup()
        dw.decode_shared_prefix()
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        assert_close(dw.out, ref, _tol(w),
                     f"{name} shared-prefix decode, {out_dtype}, all {w.num_seqs} sequences")
        # a second run from the same plan (a model's next layer) gives the same bits
        first = dw.out.clone()
        dw.shared_prefix_plan()
        dw.decode_shared_prefix_run()
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        assert torch.equal(_bits(dw.out), _bits(first))
        del dw
        torch.cuda.empty_cache()


def test_fullsize_every_sequence_counted(full):
    """The oracle's output covers every sequence and head (no sampling)."""
    name, w, ref, _, _ = full
    assert ref.shape == (w.num_seqs, w.num_heads, w.head_dim)
    assert np.all(np.isfinite(ref))
    assert np.all(np.abs(ref).sum(axis=2) > 0), f"{name}: an all-zero oracle row"
