"""decode_attn_paged_static: the entry point for callers that cannot allocate
device memory (an allocator or memory-pool callback, a plugin whose host owns
every device allocation, a loop that forbids allocation after start-up). It
uses the library's built-in scratch array instead of a caller workspace.

These tests call it through the C ABI and check it against decode_attn_paged
(which takes a workspace) and against the fp64 oracle on two calls in a row,
since every call shares, and leaves behind, the same scratch array. This file
is collected last so that a run that stops at the first failure has run every
other test first.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import binding, inputs
from paged_gqa_decode_head_gb300.runner import bf16_bits, to_device_bf16, to_device_i32
from parity_util import assert_bf16_close

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)
ATOL_F32 = 2e-3


def _case(seed, ctx, Hq=16, Hkv=8, P=16):
    kv = inputs.paged_kv(seed, ctx, Hkv=Hkv, page_size=P)
    q = inputs.query(seed, len(ctx), Hq)
    dev = "cuda"
    return dict(q=to_device_bf16(q, dev), kc=to_device_bf16(kv.k_cache, dev), vc=to_device_bf16(kv.v_cache, dev),
                bt=to_device_i32(kv.block_table, dev), ctx=to_device_i32(kv.context_lens, dev), B=len(ctx),
                Hq=Hq, Hkv=Hkv, P=P, max_pages=kv.max_pages, num_pages=kv.num_pages, host=(kv, q))


def _with_workspace(c, np_):
    ws = torch.zeros(max(16, pg.decode_attn_workspace_size(c["B"], c["Hq"], c["Hkv"], 128, c["P"], c["max_pages"],
                                                           np_)), dtype=torch.uint8, device="cuda")
    of = torch.empty((c["B"], c["Hq"], 128), dtype=torch.float32, device="cuda")
    ob = torch.empty((c["B"], c["Hq"], 128), dtype=torch.bfloat16, device="cuda")
    pg.decode_attn_paged(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"], SCALE, out_f32=of, out_bf16=ob, workspace=ws,
                         num_partitions=np_)
    return of, ob


def _static_via_c_abi(c, np_):
    lib = binding.load_library()
    of = torch.full((c["B"], c["Hq"], 128), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.full((c["B"], c["Hq"], 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.decode_attn_paged_static(
        c["q"].data_ptr(), c["kc"].data_ptr(), c["vc"].data_ptr(), c["bt"].data_ptr(), c["ctx"].data_ptr(), c["B"],
        c["Hq"], c["Hkv"], 128, c["P"], c["max_pages"], c["num_pages"], ctypes.c_float(SCALE), np_,
        of.data_ptr(), ob.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.pgqa_last_error()
    return of, ob


def test_static_scratch_matches_workspace_path_on_two_calls_in_a_row():
    # The first call (B * Hkv = 32 partition tickets, 256 bytes with their
    # alignment) leaves partition maxima at bytes 256.. of the array; the
    # second (B * Hkv = 128 tickets, 512 bytes) finds them where its tickets
    # go, so it is only right if the entry point clears its tickets first.
    # A third shape, one sequence over a few partitions, runs twice more.
    rng = np.random.default_rng(203)
    first = _case(200, [3000, 17, 1025, 64])
    second = _case(201, rng.integers(1, 2048, size=16).tolist())
    third = _case(204, [1500])
    for c, np_ in ((first, 6), (second, 4), (third, 5), (third, 5)):
        of_s, ob_s = _static_via_c_abi(c, np_)
        of_w, ob_w = _with_workspace(c, np_)
        torch.cuda.synchronize()
        # the same kernels at the same partition count: the same bits
        assert torch.equal(of_s, of_w)
        assert torch.equal(ob_s.view(torch.int16), ob_w.view(torch.int16))
        kv, q = c["host"]
        ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
        assert np.abs(of_s.cpu().numpy() - ref).max() <= ATOL_F32
        assert_bf16_close(bf16_bits(ob_s), oracle.round_bf16(ref))
    assert pg.device_error_flags() == 0


def test_static_scratch_refuses_sizes_beyond_its_array():
    c = _case(202, [64])
    lib = binding.load_library()
    # B * Hq * NP * (128 + 2) * 4 bytes far above the built-in array
    big_b, big_hq, big_np = 1, 64, 4096
    need = pg.decode_attn_workspace_size(big_b, big_hq, 8, 128, 16, 65536, big_np)
    assert need > binding.STATIC_SCRATCH_BYTES
    rc = lib.decode_attn_paged_static(c["q"].data_ptr(), c["kc"].data_ptr(), c["vc"].data_ptr(), c["bt"].data_ptr(),
                                      c["ctx"].data_ptr(), big_b, big_hq, 8, 128, 16, 65536, c["num_pages"],
                                      ctypes.c_float(SCALE), big_np, None, None, None)
    assert rc == -4
    assert b"built-in" in lib.pgqa_last_error()
