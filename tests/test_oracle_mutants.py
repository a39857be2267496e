"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them.  The mutants are built from oracle.c on the CPU into
a temporary directory; the real oracle is never modified."""
import os

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (description, text in oracle.c, replacement)
MUTANTS = [
    ("gather row uses block index", "(size_t)(j % BS)) * D;", "(size_t)(j / BS)) * D;"),
    ("interleaved GQA mapping", "g = h / group;", "g = h % job->num_kv_heads;"),
    ("scale dropped", "z[j] = scale * dot;", "z[j] = dot;"),
    ("softmax of negated scores", "z[j] = exp(z[j] - zmax);", "z[j] = exp(zmax - z[j]);"),
    ("missing normalisation", "double p = z[j] / denom;", "double p = z[j];"),
    ("pool axes transposed", "(((size_t)pb * Hkv + g) * BS + (size_t)(j % BS)) * D",
     "(((size_t)pb * BS + (size_t)(j % BS)) * Hkv + g) * D"),
    ("block table row ignored", "job->block_tables[(size_t)s * job->max_blocks_per_seq + lb]",
     "job->block_tables[lb]"),
    ("last context token dropped", "oracle_attention_contiguous(o, q, K, V, ctx, D, job->scale)",
     "oracle_attention_contiguous(o, q, K, V, ctx > 1 ? ctx - 1 : ctx, D, job->scale)"),
    ("bf16 widened with the wrong shift", "uint32_t w = (uint32_t)h << 16;",
     "uint32_t w = (uint32_t)h << 15;"),
    ("query row of the wrong head", "((size_t)s * job->num_heads + h) * D + d)",
     "((size_t)s * job->num_heads + g) * D + d)"),
    ("K used in place of V", "out[d] += p * V[(size_t)j * head_dim + d];",
     "out[d] += p * K[(size_t)j * head_dim + d];"),
    ("cache write row from block index", "off = slot % block_size;", "off = slot / block_size % block_size;"),
    ("cache write keys into both pools",
     "memcpy((char *)v_pool + dst, (const char *)value + src, row_bytes);",
     "memcpy((char *)v_pool + dst, (const char *)key + src, row_bytes);"),
    ("cache write ignores kv head", "size_t src = ((size_t)t * num_kv_heads + h) * row_bytes;",
     "size_t src = ((size_t)t * num_kv_heads) * row_bytes;"),
]


def _pin_suite():
    """Every pin of the oracle, as zero-argument callables."""
    calls = []
    for name in ["paged_gather_uniform.json", "paged_two_token_softmax.json", "paged_gqa_grouping.json"]:
        calls.append(lambda n=name: pins.test_golden_paged_decode(n))
    calls += [pins.test_golden_reshape_and_cache, pins.test_identical_keys_give_mean_of_values,
              pins.test_single_token_returns_its_value, pins.test_zero_scale_gives_mean_of_values,
              pins.test_two_keys_logistic_closed_form, pins.test_empty_context_is_zero,
              pins.test_tiny_f32_workload_matches_brute_force,
              pins.test_reshape_then_gather_round_trip_and_untouched_bytes,
              pins.test_reshape_negative_slot_is_skipped_bf16,
              pins.test_shared_prefix_equals_unshared_copies]
    for hot in (0, 5, 12):
        calls.append(lambda h=hot: pins.test_one_hot_key_closed_form(h))
    for dt in ("f32", "bf16"):
        for heads in ((4, 4), (4, 2)):
            calls.append(lambda d=dt, hh=heads: pins.test_matches_decimal_brute_force(d, hh))
    return calls


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, desc, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    caught = 0
    with oracle.use_library(lib):
        for call in _pin_suite():
            try:
                call()
            except (AssertionError, ValueError):
                caught += 1
    assert caught > 0, f"no pin caught the mutant: {desc}"
