"""Register and spill budgets of the main decode kernels, read from the
compiler's resource report (`-Xptxas -v`) on the CPU.

The launch code counts on them: the plain decode's automatic partition
assumes three resident CTAs per SM (128 threads each, so at most 170
registers a thread), and the shared-prefix decode sizes its persistent grid
for two (255).  A source change that pushes a kernel over its budget, or
makes it spill, keeps every result right and only shows as a slower
decode; this catches it before any GPU run.
"""
import os
import re
import shutil
import subprocess

import pytest

from paged_kv_cache_249_gb300 import build

ENTRY = re.compile(r"Compiling entry function '([^']+)'")
USED = re.compile(r"Used (\d+) registers")
SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")


def _resources(source: str) -> dict:
    """Mangled kernel name -> (registers, spill store bytes) for one unit."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is not available")
    out = os.path.join(build.BUILD_DIR, "resources_" + os.path.basename(source) + ".o")
    os.makedirs(build.BUILD_DIR, exist_ok=True)
    res = subprocess.run([nvcc, *build.ARCH, *build.NVCC_FLAGS, "-Xptxas", "-v", "-c",
                          os.path.join(build.CSRC, source), "-o", out],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    found, name, spill = {}, None, 0
    for line in res.stderr.splitlines():
        m = ENTRY.search(line)
        if m:
            name, spill = m.group(1), 0
            continue
        m = SPILL.search(line)
        if m and name:
            spill = int(m.group(1))
        m = USED.search(line)
        if m and name:
            found[name] = (int(m.group(1)), spill)
            name = None
    return found


def _pick(found: dict, *parts: str) -> tuple:
    hits = [v for k, v in found.items() if all(p in k for p in parts)]
    assert len(hits) == 1, (parts, sorted(found))
    return hits[0]


def test_plain_decode_fits_three_ctas_per_sm():
    found = _resources("decode_bf16_d128.cu")
    # template arguments <T, D, BS, GP, MMA, RUNS> as the mangled name spells them
    for gp, mma, runs in (("8", "1", "0"), ("16", "1", "0"), ("1", "0", "0"), ("4", "0", "0"),
                          ("8", "1", "1")):
        args = f"Li128ELi16ELi{gp}ELb{mma}ELb{runs}E"
        regs, spill = _pick(found, "paged_decode_kernel", "nv_bfloat16", args)
        assert regs <= 170 and spill == 0, (args, regs, spill)


def test_fp32_tensor_core_decode_fits_three_ctas_per_sm():
    found = _resources("decode_f32_d128.cu")
    for gp in ("8", "16"):
        regs, spill = _pick(found, "paged_decode_kernel", f"Li128ELi16ELi{gp}ELb1ELb0E")
        assert regs <= 170 and spill == 0, (gp, regs, spill)


def test_shared_prefix_decode_fits_two_ctas_per_sm_without_spills():
    found = _resources("shared_prefix_d128.cu")
    regs, spill = _pick(found, "shared_prefix_decode_kernel")
    assert regs <= 255 and spill == 0, (regs, spill)
