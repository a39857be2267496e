"""Decode steps captured in CUDA graphs and replayed.

A serving loop replays one captured decode step per token, so every call of
the path must be capturable: it only enqueues work on the caller's stream
(programmatic dependent launches become graph edges), allocates nothing and
never synchronises.  Each test captures a step once, then replays it with
new queries (and, for the shared-prefix path, a new plan) copied into the
captured buffers, and checks every replay against the float64 oracle.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


def _new_queries(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.q.shape, generator=g).to(w.q.dtype)


@pytest.mark.parametrize("dtype,H,Hkv,pt", [("bf16", 32, 8, 64), ("bf16", 16, 16, 0),
                                             ("f32", 8, 2, 128)])
def test_plain_decode_step_replays(dtype, H, Hkv, pt):
    w = workload.build(f"graph_{dtype}_{H}_{Hkv}", dtype=dtype,
                       context_lens=[1, 17, 300, 1025, 64, 700], num_heads=H, num_kv_heads=Hkv,
                       head_dim=128, block_size=16, data_seed=700 + H, meta_seed=710 + H)
    dw = pagedkv.DeviceWorkload(w, partition_tokens=pt)
    dw.step()  # eager warm-up: one-time kernel attribute set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dw.step()
    for rep in range(3):
        q = _new_queries(w, rep)
        dw.q.copy_(q)
        dw.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        w.q = q
        ref, _, _ = oracle_after_write(w)
        assert_close(dw.out, ref, dtype, f"replay {rep}")


def test_shared_prefix_plan_and_run_replay():
    """Plan and run captured as one step; a replay after the context lengths
    grow (one more token per sequence) re-plans from the new lengths."""
    ctx = [256 + s for s in (3, 40, 90, 0, 17, 200)] + [70, 64, 100]
    w = workload.build("graph_sp", dtype="bf16", context_lens=ctx, num_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=16, data_seed=720, meta_seed=721,
                       groups=[(6, 256), (3, 64)], max_blocks_per_seq=40)
    dw = pagedkv.DeviceWorkload(w)
    dw.shared_prefix_setup(partition_tokens=0)
    pagedkv.reshape_and_cache(dw.pool, dw.new_key, dw.new_value, dw.slot_mapping)
    dw.decode_shared_prefix()  # eager warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dw.decode_shared_prefix()
    for rep in range(3):
        q = _new_queries(w, 10 + rep)
        dw.q.copy_(q)
        dw.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pagedkv.get_device_error(dw.pool) == 0
        w.q = q
        ref, _, _ = oracle_after_write(w)
        assert_close(dw.out, ref, "bf16", f"replay {rep}")
    # shorter contexts (every sequence loses its last token; still within the
    # captured bounds): the captured plan kernel re-plans from the new lengths
    shorter = np.maximum(np.asarray(ctx) - 1, 0)
    shorter[:6] = np.maximum(shorter[:6], 256)
    shorter[6:] = np.maximum(shorter[6:], 64)
    dw.context_lens.copy_(torch.from_numpy(shorter.astype(np.int32)))
    graph.replay()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    w.context_lens = shorter.astype(np.int32)
    ref, _, _ = oracle_after_write(w)
    assert_close(dw.out, ref, "bf16", "after the contexts changed")
