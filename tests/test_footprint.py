"""Memory-footprint report: pinned by the pages' worked example."""
import json
import os

from paged_kv_cache_249_gb300 import footprint, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "naive_reservation_example.json")


def test_pages_worked_example():
    g = json.load(open(GOLDEN))
    assert footprint.naive_slots(1, g["max_context"]) - g["tokens_used"] == \
        g["expected_naive_wasted_slots"]
    paged = footprint.paged_slots([g["tokens_used"]], g["block_size"])
    assert paged == g["expected_paged_slots"]
    assert paged - g["tokens_used"] == g["expected_paged_wasted_slots"]


def test_shared_prefix_counts_prefix_once():
    # 2 groups x 3 sequences, 32-token prefix (2 blocks of 16) + 5-token suffix
    ctx = [37] * 6
    assert footprint.paged_slots(ctx, 16) == 6 * 3 * 16
    assert footprint.paged_slots(ctx, 16, shared_prefix_blocks=2, group_size=3) == \
        (6 * 3 - 2 * 2 * 2) * 16


def test_report_on_a_workload():
    w = workload.make("tiny_f32")
    r = footprint.report(w)
    assert r["tokens"] == 5 + 17 + 33 + 64
    assert r["paged_bytes"] == 10 * 16 * footprint.kv_bytes_per_token(4, 64, 4)
    assert r["naive_bytes"] == 4 * 64 * footprint.kv_bytes_per_token(4, 64, 4)
