"""Paged = contiguous, on the GPU: the same tokens read through a block table
from a shuffled pool, or from a conventional contiguous cache, give bitwise
the same attention (the block table is an indirection only: Qualiteg,
"About PagedAttention for LLM serving", the section on logical and physical
blocks; vAttention section 3.1
contrasts the two layouts)."""
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("partition", [-1, 0, 256])
@pytest.mark.parametrize("dtype,H,Hkv,D", [("bf16", 32, 8, 128), ("bf16", 16, 16, 128),
                                           ("f32", 8, 2, 128), ("f16", 32, 8, 128),
                                           ("bf16", 16, 4, 256)])
def test_contiguous_equals_paged_bitwise(dtype, H, Hkv, D, partition):
    w = workload.build("contig", dtype=dtype, context_lens=[1, 300, 17, 1024, 511], num_heads=H,
                       num_kv_heads=Hkv, head_dim=D, block_size=16, data_seed=3, meta_seed=4)
    dw = pagedkv.DeviceWorkload(w, partition_tokens=partition)
    dw.step()
    cache = pagedkv.ContiguousCache.from_paged(w, k_pool=dw.k_pool, v_pool=dw.v_pool)
    out = torch.empty_like(dw.out)
    pagedkv.contiguous_attention_decode(cache, out, dw.q, dw.context_lens, dw.max_context_len,
                                        w.scale, partition_tokens=partition,
                                        workspace=dw.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), dw.out.view(torch.int32))
    ref, _, _ = oracle_after_write(w)
    assert_close(out, ref, dtype, "contiguous")


@pytest.mark.parametrize("name", ["mha_7b", "gqa_8b"])
def test_contiguous_equals_paged_fullsize(name):
    w = workload.make(name)
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    dw.step()
    cache = pagedkv.ContiguousCache.from_paged(w, k_pool=dw.k_pool, v_pool=dw.v_pool)
    out = torch.empty_like(dw.out)
    pagedkv.contiguous_attention_decode(cache, out, dw.q, dw.context_lens, dw.max_context_len,
                                        w.scale, workspace=dw.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dw.out.view(torch.int16))


def test_contiguous_rejects_paged_calls():
    k = torch.zeros(2, 2, 32, 64, dtype=torch.bfloat16, device="cuda")
    cache = pagedkv.ContiguousCache(k, k.clone())
    with pytest.raises(pagedkv.PagedKVError):
        pagedkv.reshape_and_cache(cache, k[0, :, 0], k[0, :, 0],
                                  torch.zeros(2, dtype=torch.int64, device="cuda"))
