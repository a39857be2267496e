"""Host-side helpers of bench.py (no GPU): shape flags, launch statistics,
clock-sample summaries, algorithmic bytes and workload overrides."""
import argparse
import importlib.util
import os

import numpy as np
import pytest

from paged_kv_cache_249_gb300 import workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_shape_flags_map_to_workload_keywords(bench):
    args = argparse.Namespace(dtype="f16", block_size=64, head_dim=None, num_heads=16,
                              num_kv_heads=None, partition=-1)
    assert bench.shape_overrides(args) == {"dtype": "f16", "block_size": 64, "num_heads": 16,
                                           "partition_tokens": -1}
    none = argparse.Namespace(dtype=None, block_size=None, head_dim=None, num_heads=None,
                              num_kv_heads=None, partition=None)
    assert bench.shape_overrides(none) == {}


def test_launch_stats_mean_median_and_fractions(bench):
    ms = [0.1, 0.1, 0.4]  # milliseconds
    st = bench.launch_stats(ms, alg_bytes=1_000_000_000, peak=5000.0)
    assert st["us_mean"] == pytest.approx(200.0)
    assert st["us_median"] == pytest.approx(100.0)
    assert st["achieved_gbs"] == pytest.approx(5000.0)  # 1 GB in 200 us
    assert st["frac"] == pytest.approx(1.0)
    assert st["frac_median"] == pytest.approx(2.0)
    assert st["launches"] == 3 and st["device_seconds"] == pytest.approx(0.0006, abs=5e-4)


def test_clock_summary_counts_samples_in_the_window(bench):
    cs = object.__new__(bench.ClockSampler)
    cs.proc = object()  # a running sampler (never touched by summary)
    row = lambda mhz, pc="Not Active": ["t", str(mhz), "2070", "900", "0x0",  # noqa: E731
                                         "Not Active", "Not Active", "Not Active", pc]
    cs.samples = [(0.5, row(1000)), (1.0, row(2070)), (1.1, row(2000)),
                  (1.2, row(2070, "Active")), (3.0, row(500))]
    s = cs.summary(0.9, 1.3)
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    # a window with no sample falls back to the nearest one and says so
    s = cs.summary(2.8, 2.9)  # nearest sample: t = 3.0
    assert s["samples"] == 1 and s["sm_mhz"] == 500.0 and "nearest" in s["window"]
    cs.proc = None
    assert bench.ClockSampler.summary(cs, 0, 1)["reasons"] == ["unavailable"]


def test_algorithmic_bytes_of_the_tiny_workload(bench):
    w = workload.make("tiny_f32")
    ab = bench.algorithmic_bytes(w)
    ctx = np.array([5, 17, 33, 64])
    assert ab["kv_logical"] == ab["kv_unique"] == int(ctx.sum()) * 4 * 64 * 2 * 4
    assert ab["table"] == int(np.sum(-(-ctx // 16))) * 4
    assert ab["q"] == 4 * 4 * 64 * 4 and ab["out"] == 4 * 4 * 64 * 2
    assert ab["decode_launch"] == ab["kv_unique"] + ab["q"] + ab["out"] + ab["table"] + 4 * 4


def test_block_size_override_keeps_lengths_and_sizes_the_table():
    base = workload.make("tiny_f32")
    w = workload.make("tiny_f32", block_size=32)
    assert np.array_equal(w.context_lens, base.context_lens)
    assert w.block_size == 32 and w.max_blocks_per_seq == 2  # 64 tokens in 32-token blocks
    for s, c in enumerate(w.context_lens):
        nb = -(-int(c) // 32)
        assert np.all(w.block_tables[s, :nb] >= 0) and np.all(w.block_tables[s, nb:] == -1)


def test_shared_prefix_shapes_the_bench_routes(bench):
    assert bench.shared_prefix_supported(workload.make("tiny_f32"))  # fp32, head size 64
    w16 = workload.make("tiny_f32", dtype="bf16", head_dim=128)
    assert bench.shared_prefix_supported(w16)
    assert bench.shared_prefix_supported(workload.make("tiny_f32", dtype="bf16", head_dim=256))
    assert not bench.shared_prefix_supported(workload.make("tiny_f32", head_dim=256))  # fp32, 256
    assert not bench.shared_prefix_supported(workload.make("tiny_f32", block_size=8))


def test_kernel_source_lists_name_existing_files(bench):
    """The files whose hash dates each stored DRAM-traffic record exist, and
    the hash is a function of their contents alone."""
    csrc = os.path.join(ROOT, "paged_kv_cache_249_gb300", "csrc")
    for family, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.isfile(os.path.join(csrc, f)), (family, f)
        assert bench.kernel_source_hash(family) == bench.kernel_source_hash(family)
    for (name, family), rec in bench.NCU_TRAFFIC.items():
        assert family in bench.KERNEL_SOURCES and rec["bytes"] > 0 and len(rec["src"]) == 16
