"""Full-size decode workloads, in the launch configuration the benchmark
times (bf16 output, automatic or workload-given partitioning, automatic
compute path), checked on sampled sequences against the float64 oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_249_gb300 import pagedkv, workload
from tests.gpu_helpers import assert_close, oracle_after_write

pytestmark = pytest.mark.gpu


def _sample(w, k=6, seed=0):
    ctx = w.context_lens
    picks = {0, w.num_seqs - 1, int(np.argmax(ctx)), int(np.argmin(ctx))}
    rng = np.random.default_rng(seed)
    while len(picks) < min(k, w.num_seqs):
        picks.add(int(rng.integers(0, w.num_seqs)))
    if w.group_size > 1:  # two members of one shared-prefix group
        picks.update({w.group_size, w.group_size + 1})
    return sorted(picks)


@pytest.mark.parametrize("name", ["mha_7b", "gqa_8b", "shared_prefix", "long_ctx"])
def test_fullsize_sampled(name):
    w = workload.make(name)
    dw = pagedkv.DeviceWorkload(w, out_dtype=torch.bfloat16)
    dw.step()
    torch.cuda.synchronize()
    assert pagedkv.get_device_error(dw.pool) == 0
    seqs = _sample(w)
    ref, _, _ = oracle_after_write(w, seqs)
    out_bf16 = dw.out[torch.tensor(seqs, device=dw.out.device)]
    assert_close(out_bf16, ref, "bf16", f"{name} bf16 output")
    # same launch with fp32 output (the pool already holds the new tokens)
    dw32 = pagedkv.DeviceWorkload(w, out_dtype=torch.float32)
    dw32.step()
    torch.cuda.synchronize()
    out32 = dw32.out[torch.tensor(seqs, device=dw32.out.device)]
    assert_close(out32, ref, "bf16", f"{name} fp32 output")
    # the bf16 output is the fp32 output rounded once
    assert torch.equal(out32.to(torch.bfloat16).cpu().view(torch.int16),
                       out_bf16.cpu().view(torch.int16))
