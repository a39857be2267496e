"""The C-ABI library loads, exports every function include/pagedkv.h declares,
agrees with the binding on struct layout, and rejects bad arguments on the
host before touching the GPU.  No test here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_249_gb300 import build as pkv_build
from paged_kv_cache_249_gb300 import pagedkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pagedkv.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = _declared_functions()
    assert set(names) == set(pagedkv.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pagedkv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), f"{n} not exported as a C symbol"


def test_struct_layout_matches_c(tmp_path, lib):
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pagedkv.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu\\n", sizeof(pkv_pool), '
                   'offsetof(pkv_pool, k_pool), offsetof(pkv_pool, dev_error), '
                   'offsetof(pkv_pool, tma));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    P = pagedkv.pkv_pool
    assert got == [ctypes.sizeof(P), P.k_pool.offset, P.dev_error.offset, P.tma.offset]


def test_header_compiles_as_c_and_cxx(tmp_path):
    for cc, ext in (("gcc", "c"), ("g++", "cpp")):
        src = tmp_path / f"inc.{ext}"
        src.write_text('#include "pagedkv.h"\nint f(void){return (int)PKV_OK;}\n')
        subprocess.run([cc, "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c",
                        str(src), "-o", str(tmp_path / f"inc_{ext}.o")], check=True)


def test_sizes_and_strings(lib):
    assert lib.pkv_version() >= 100
    assert lib.pkv_pool_bytes(10, 16, 8, 128, pagedkv.BF16) == 10 * 16 * 8 * 128 * 2
    assert lib.pkv_pool_bytes(10, 16, 8, 64, pagedkv.F32) == 10 * 16 * 8 * 64 * 4
    assert lib.pkv_pool_bytes(0, 16, 8, 64, pagedkv.F32) == 0
    assert lib.pkv_pool_bytes(10, 16, 8, 128, pagedkv.F16) == 10 * 16 * 8 * 128 * 2
    assert lib.pkv_pool_bytes(10, 16, 8, 128, 3) == 0  # no such dtype
    for s in range(6):
        assert lib.pkv_status_string(s)
    # split-K partials: S*H*P*(D+1) floats, each part rounded to 256 bytes
    S, H, D, ctx, pt = 8, 64, 128, 131072, 512
    P = ctx // pt
    o = S * H * P * D * 4
    lse = -(-(S * H * P * 4) // 256) * 256
    assert lib.pkv_decode_workspace_bytes(S, H, D, ctx, pt) == o + lse
    assert lib.pkv_decode_workspace_bytes(S, H, D, ctx, 0) == o + lse  # auto = 512
    assert lib.pkv_decode_workspace_bytes(S, H, D, ctx, -1) == 0
    assert lib.pkv_decode_workspace_bytes(S, H, D, 512, 0) == 0       # fits one partition


def _fake_pool(**kw):
    """A descriptor that passes the 'initialised' check but points nowhere;
    only used for calls that must fail validation before any CUDA call."""
    p = pagedkv.pkv_pool()
    p.magic = 0x504B5631
    p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim = 64, 16, 2, 128
    p.dtype = pagedkv.BF16
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _decode(lib, pool, **kw):
    args = dict(out=0x1000, out_dtype=pagedkv.F32, query=0x2000, num_seqs=4, num_heads=8,
                num_kv_heads=2, block_tables=0x3000, max_blocks=8, context_lens=0x4000,
                max_ctx=128, scale=0.1, partition=0, ws=None, ws_bytes=0, flags=0, stream=None)
    args.update(kw)
    return lib.pkv_paged_attention_decode(
        ctypes.byref(pool) if pool is not None else None, args["out"], args["out_dtype"],
        args["query"], args["num_seqs"], args["num_heads"], args["num_kv_heads"],
        args["block_tables"], args["max_blocks"], args["context_lens"], args["max_ctx"],
        args["scale"], args["partition"], args["ws"], args["ws_bytes"], args["flags"],
        args["stream"])


def test_decode_rejects_bad_arguments_on_host(lib):
    E, U = pagedkv.ERR_INVALID_ARG, pagedkv.ERR_UNSUPPORTED
    pool = _fake_pool()
    assert _decode(lib, None) == E                                   # no pool
    assert _decode(lib, pagedkv.pkv_pool()) == E                     # not initialised
    assert _decode(lib, pool, num_kv_heads=4, num_heads=8) == E      # != pool heads
    assert _decode(lib, pool, num_heads=7) == E                      # not a multiple
    assert _decode(lib, pool, num_heads=34) == U                     # group 17 > 16
    assert _decode(lib, pool, out=0) == E                            # null output
    assert _decode(lib, pool, query=0x2004) == E                     # misaligned
    assert _decode(lib, pool, partition=24) == E                     # not a block multiple
    assert _decode(lib, pool, partition=16384) == E                  # above the maximum
    assert _decode(lib, pool, out_dtype=7) == E
    assert _decode(lib, pool, flags=9) == E
    assert _decode(lib, pool, scale=float("nan")) == E
    assert _decode(lib, pool, max_blocks=0) == E
    # fp32 tensor-core tiles (TF32) are built up to head size 128
    assert _decode(lib, _fake_pool(dtype=pagedkv.F32, head_dim=256), flags=pagedkv.PATH_MMA) == U
    assert _decode(lib, pool, num_seqs=0) == pagedkv.OK              # nothing to do


def test_pool_init_and_cache_write_reject_bad_arguments(lib):
    E, U = pagedkv.ERR_INVALID_ARG, pagedkv.ERR_UNSUPPORTED
    p = pagedkv.pkv_pool()
    init = lib.pkv_block_pool_init
    assert init(None, 8, 16, 2, 128, pagedkv.BF16, 0x1000, 0x2000, None, 0, None) == E
    assert init(ctypes.byref(p), 8, 16, 2, 128, pagedkv.BF16, 0, 0x2000, None, 0, None) == E
    # block sizes: 16, 32, 64, 128 or 256 tokens (the page's range of roughly 16 to 256)
    for bs in (8, 24, 48, 96, 512):
        assert init(ctypes.byref(p), 8, bs, 2, 128, pagedkv.BF16, 0x1000, 0x2000, None, 0,
                    None) == U, bs
    assert init(ctypes.byref(p), 8, 16, 2, 96, pagedkv.BF16, 0x1000, 0x2000, None, 0, None) == U
    assert init(ctypes.byref(p), 8, 16, 2, 128, 5, 0x1000, 0x2000, None, 0, None) == E
    assert init(ctypes.byref(p), 8, 16, 2, 128, pagedkv.BF16, 0x1008, 0x2000, None, 0, None) == E
    assert p.magic == 0  # nothing was filled in
    rc = lib.pkv_reshape_and_cache
    assert rc(ctypes.byref(p), 0x1000, 0x2000, 0x3000, 4, None) == E  # pool not initialised
    fp = _fake_pool()
    assert rc(ctypes.byref(fp), 0, 0x2000, 0x3000, 4, None) == E
    assert rc(ctypes.byref(fp), 0x1000, 0x2000, 0x3004, 4, None) == E  # misaligned slots
    assert rc(ctypes.byref(fp), 0x1000, 0x2000, 0x3000, -1, None) == E
    assert rc(ctypes.byref(fp), 0x1000, 0x2000, 0x3000, 0, None) == pagedkv.OK


def test_block_table_upload_checks_entries_on_host(lib):
    import numpy as np
    host = np.array([[0, 5, -1], [7, 8, 9]], dtype=np.int32)
    up = lib.pkv_block_table_upload
    assert up(0x1000, host.ctypes.data, 2, 3, 9, None) == pagedkv.ERR_INVALID_ARG  # 9 >= 9
    assert up(0, host.ctypes.data, 2, 3, 0, None) == pagedkv.ERR_INVALID_ARG
    assert up(0x1000, host.ctypes.data, 2, 0, 0, None) == pagedkv.ERR_INVALID_ARG
    assert up(0x1000, host.ctypes.data, 0, 3, 0, None) == pagedkv.OK


def _sp_decode(lib, pool, **kw):
    args = dict(out=0x1000, out_dtype=pagedkv.F32, query=0x2000, num_seqs=4, num_heads=8,
                num_kv_heads=2, block_tables=0x3000, max_blocks=8, context_lens=0x4000,
                max_ctx=128, scale=0.1, group_starts=0x5000, prefix_lens=0x6000, num_groups=2,
                max_prefix=64, partition=0, ws=0x7000, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.pkv_paged_attention_decode_shared_prefix(
        ctypes.byref(pool) if pool is not None else None, args["out"], args["out_dtype"],
        args["query"], args["num_seqs"], args["num_heads"], args["num_kv_heads"],
        args["block_tables"], args["max_blocks"], args["context_lens"], args["max_ctx"],
        args["scale"], args["group_starts"], args["prefix_lens"], args["num_groups"],
        args["max_prefix"], args["partition"], args["ws"], args["ws_bytes"], args["stream"])


def test_shared_prefix_decode_rejects_bad_arguments_on_host(lib):
    E, U = pagedkv.ERR_INVALID_ARG, pagedkv.ERR_UNSUPPORTED
    pool = _fake_pool()
    assert _sp_decode(lib, None) == E                                # no pool
    assert _sp_decode(lib, pagedkv.pkv_pool()) == E                  # not initialised
    assert _sp_decode(lib, pool, num_groups=0) == E                  # groups must cover the batch
    assert _sp_decode(lib, pool, num_groups=5) == E                  # more groups than sequences
    assert _sp_decode(lib, pool, group_starts=0) == E
    assert _sp_decode(lib, pool, prefix_lens=0x6002) == E            # misaligned
    assert _sp_decode(lib, pool, max_prefix=-1) == E
    assert _sp_decode(lib, pool, partition=24) == E                  # not a block multiple
    assert _sp_decode(lib, pool, num_kv_heads=4) == E                # != pool heads
    assert _sp_decode(lib, pool, scale=float("inf")) == E
    assert _sp_decode(lib, _fake_pool(dtype=pagedkv.F32, head_dim=256)) == U  # fp32 up to 128
    # a 256-wide head passes the shape checks (here it stops at the missing workspace)
    assert _sp_decode(lib, _fake_pool(head_dim=256), ws_bytes=0) == pagedkv.ERR_WORKSPACE
    assert _sp_decode(lib, pool, num_heads=34) == U                  # group 17 > 16
    assert _sp_decode(lib, pool, num_seqs=0) == pagedkv.OK           # nothing to do


def test_shared_prefix_workspace_bytes(lib):
    """Header, per-sequence counts and sharing records, the work list, and
    the partials: one slot per prefix part (sized for 512-token parts, the
    shortest the automatic choice takes) and per own part (256 tokens by
    default) of the longest sequence."""
    r = lambda x: -(-x // 256) * 256  # noqa: E731

    def expect(S, H, D, maxc, maxp, pt):
        mp = min(maxp, maxc)
        if pt < 0:
            pp, ps = int(mp > 0), int(maxc > 0)
        else:
            ptp, pts = (pt, pt) if pt > 0 else (512, 256)
            pp, ps = -(-mp // ptp), -(-maxc // pts)
        slots = max(pp + ps, 1)
        return (256 + r(S * 4) + r(S * 8) + r(S * slots * 32) + r(S * H * slots * 4) +
                r(S * H * slots * D * 4))

    f = lib.pkv_shared_prefix_workspace_bytes
    for S, H, D, maxc, maxp, pt in [(256, 32, 128, 4608, 4096, 0), (8, 64, 128, 131072, 0, 0),
                                    (3, 4, 64, 100, 48, 32), (5, 8, 128, 2000, 1024, -1),
                                    (2, 2, 64, 64, 999, 0)]:
        assert f(S, H, D, maxc, maxp, pt) == expect(S, H, D, maxc, maxp, pt), (S, maxc, maxp, pt)
    assert f(0, 8, 128, 100, 0, 0) == 0
    assert f(4, 8, 128, 100, -1, 0) == 0


def test_shared_prefix_plan_and_run_reject_bad_arguments_on_host(lib):
    E, U = pagedkv.ERR_INVALID_ARG, pagedkv.ERR_UNSUPPORTED
    pool = _fake_pool()

    def plan(p, **kw):
        a = dict(S=4, H=8, Hkv=2, MB=8, cl=0x4000, maxc=128, gs=0x5000, pl=0x6000, ng=2, maxp=64,
                 pt=0, ws=0x7000, wsb=1 << 20)
        a.update(kw)
        return lib.pkv_shared_prefix_plan(
            ctypes.byref(p) if p is not None else None, a["S"], a["H"], a["Hkv"], a["MB"],
            a["cl"], a["maxc"], a["gs"], a["pl"], a["ng"], a["maxp"], a["pt"], a["ws"], a["wsb"],
            None)

    def run(p, **kw):
        a = dict(out=0x1000, dt=pagedkv.F32, q=0x2000, S=4, H=8, Hkv=2, bt=0x3000, MB=8,
                 maxc=128, scale=0.1, maxp=64, pt=0, ws=0x7000, wsb=1 << 20)
        a.update(kw)
        return lib.pkv_paged_attention_decode_shared_prefix_run(
            ctypes.byref(p) if p is not None else None, a["out"], a["dt"], a["q"], a["S"], a["H"],
            a["Hkv"], a["bt"], a["MB"], a["maxc"], a["scale"], a["maxp"], a["pt"], a["ws"],
            a["wsb"], None)

    assert plan(None) == E
    assert plan(pool, ng=0) == E
    assert plan(pool, cl=0) == E
    assert plan(pool, gs=0x5002) == E
    assert plan(pool, pt=24) == E
    assert plan(pool, wsb=16) == pagedkv.ERR_WORKSPACE
    assert plan(_fake_pool(dtype=pagedkv.F32, head_dim=256)) == U  # fp32 up to head size 128
    assert plan(pool, S=0) == pagedkv.OK
    assert run(None) == E
    assert run(pool, out=0) == E
    assert run(pool, q=0x2008) == E
    assert run(pool, scale=float("nan")) == E
    assert run(pool, dt=9) == E
    assert run(pool, H=34) == U
    assert run(pool, ws=0x7010) == E                                  # not 256-byte aligned
    assert run(pool, S=0) == pagedkv.OK


def test_bounded_wait_check_rejects_bad_arguments_on_host(lib):
    E = pagedkv.ERR_INVALID_ARG
    chk = lib.pkv_check_bounded_wait
    assert chk(None, 1000000, None) == E
    assert chk(ctypes.byref(_fake_pool()), 1000000, None) == E      # pool without an error word
    fp = _fake_pool(dev_error=0x5000)
    for limit in (0, 999, 2000000001, -5):
        assert chk(ctypes.byref(fp), limit, None) == E, limit
