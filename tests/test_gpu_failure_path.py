"""The failure path of a wait that never completes, exercised without a
fault: a kernel waits on an mbarrier that nothing arrives on, gives up after
its limit, raises PGQA_DEVERR_WAIT_TIMEOUT and returns; the context stays
usable and the next calls are correct."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import binding, inputs
from paged_gqa_decode_head_gb300.runner import to_device_bf16, to_device_i32

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)


def test_bounded_wait_gives_up_and_context_stays_usable():
    pg.device_error_flags(clear=True)
    binding.selftest_wait_timeout()
    flags = pg.device_error_flags(clear=True)
    assert flags & binding.DEVERR_WAIT_TIMEOUT
    assert pg.device_error_flags() == 0  # cleared

    kv = inputs.paged_kv(590, [300, 45], Hkv=8, page_size=16)
    q = inputs.query(590, 2, 16, 128)
    ws = torch.zeros(max(16, pg.decode_attn_workspace_size(2, 16, 8, 128, 16, kv.max_pages, 3)), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((2, 16, 128), dtype=torch.float32, device="cuda")
    pg.decode_attn_paged(to_device_bf16(q, "cuda"), to_device_bf16(kv.k_cache, "cuda"),
                         to_device_bf16(kv.v_cache, "cuda"), to_device_i32(kv.block_table, "cuda"),
                         to_device_i32(kv.context_lens, "cuda"), SCALE, out_f32=out, workspace=ws, num_partitions=3)
    torch.cuda.synchronize()
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
    assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
    assert pg.device_error_flags() == 0
