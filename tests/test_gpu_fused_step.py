"""GPU parity of decode_step_paged, the fused one-launch decode step: the
prologue (Q/K RMSNorm, RoPE, K/V append) and the paged attention together,
against the oracle's chain and against the two separate entry points."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import binding, inputs
from paged_gqa_decode_head_gb300.runner import bf16_bits, to_device_bf16, to_device_i32
from parity_util import assert_bf16_close, walked

pytestmark = pytest.mark.gpu

ATOL_F32 = 2e-3
THETA = 1e6
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(autouse=True)
def _clean_flags():
    pg.device_error_flags(clear=True)
    yield


def _device_case(kv, tok):
    dev = "cuda"
    return dict(q=to_device_bf16(tok.q, dev), k=to_device_bf16(tok.k, dev), v=to_device_bf16(tok.v, dev),
                gq=to_device_bf16(tok.gamma_q, dev), gk=to_device_bf16(tok.gamma_k, dev),
                ctx=to_device_i32(kv.context_lens, dev), bt=to_device_i32(kv.block_table, dev),
                kc=to_device_bf16(kv.k_cache, dev), vc=to_device_bf16(kv.v_cache, dev))


def _workspace(kv, Hq, Hkv, num_partitions):
    n = pg.decode_attn_workspace_size(len(kv.context_lens), Hq, Hkv, 128, kv.page_size, kv.max_pages, num_partitions)
    return torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")


def run_fused(kv, tok, num_partitions=0):
    c = _device_case(kv, tok)
    B, Hq, D = tok.q.shape
    Hkv = tok.k.shape[1]
    q_out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    of = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pg.decode_step_paged(c["q"], c["k"], c["v"], c["gq"], c["gk"], c["ctx"], c["bt"], c["kc"], c["vc"], SCALE, THETA,
                         q_out=q_out, out_f32=of, out_bf16=ob, workspace=_workspace(kv, Hq, Hkv, num_partitions),
                         num_partitions=num_partitions)
    torch.cuda.synchronize()
    return dict(q_out=bf16_bits(q_out), kc=bf16_bits(c["kc"]), vc=bf16_bits(c["vc"]), of=of.cpu().numpy(),
                ob=bf16_bits(ob))


def run_unfused(kv, tok, num_partitions=0):
    c = _device_case(kv, tok)
    B, Hq, D = tok.q.shape
    Hkv = tok.k.shape[1]
    q_out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    of = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ob = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    pg.qk_norm_rope_append(c["q"], c["k"], c["v"], c["gq"], c["gk"], c["ctx"], c["bt"], c["kc"], c["vc"], q_out,
                           kv.page_size, THETA)
    pg.decode_attn_paged(q_out, c["kc"], c["vc"], c["bt"], c["ctx"], SCALE, out_f32=of, out_bf16=ob,
                         workspace=_workspace(kv, Hq, Hkv, num_partitions), num_partitions=num_partitions)
    torch.cuda.synchronize()
    return dict(q_out=bf16_bits(q_out), kc=bf16_bits(c["kc"]), vc=bf16_bits(c["vc"]), of=of.cpu().numpy(),
                ob=bf16_bits(ob))


def check_fused(kv, tok, num_partitions=0):
    got = run_fused(kv, tok, num_partitions)
    q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                       kv.context_lens, kv.block_table, kv.k_cache, kv.v_cache,
                                                       kv.page_size, THETA)
    assert_bf16_close(got["q_out"], q_ref, "q_out")
    assert np.array_equal(got["vc"], vc_ref)  # V appended bit for bit, nothing else written
    changed = np.any(got["kc"] != kv.k_cache, axis=-1) | np.any(kc_ref != kv.k_cache, axis=-1)
    assert np.array_equal(got["kc"][~changed], kv.k_cache[~changed])
    assert_bf16_close(got["kc"], kc_ref, "appended K")
    # the whole chain against the oracle's chain (fp32 bar); the attention
    # alone on the step's own q_out and cache (which may differ from the
    # oracle's by 1 bf16 ulp, checked above) for the bf16 bar
    ref = oracle.decode_attention(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
    assert np.isfinite(got["of"]).all()
    assert np.abs(got["of"] - ref).max() <= ATOL_F32
    own = oracle.decode_attention(got["q_out"], got["kc"], got["vc"], kv.block_table, kv.context_lens, SCALE)
    assert np.abs(got["of"] - own).max() <= ATOL_F32
    assert_bf16_close(got["ob"], oracle.round_bf16(own), "out_bf16")
    assert pg.device_error_flags() == 0
    return got


@pytest.mark.parametrize("T", [1, 2, 3, 8, 15, 16, 17, 31, 32, 33, 512, 513])
def test_fused_step_small_and_boundary_contexts(T):
    kv = inputs.paged_kv(300 + T, [T], Hkv=8, page_size=16)
    tok = inputs.new_token(300 + T, 1, 16, 8)
    check_fused(kv, tok)


@pytest.mark.parametrize("num_partitions", [0, 1, 3, 100])
@pytest.mark.parametrize("P", [16, 64])
def test_fused_step_ragged_batch(num_partitions, P):
    ctx = [1, 17, 300, 4097, 2000]
    kv = inputs.paged_kv(320 + P, ctx, Hkv=8, page_size=P)
    tok = inputs.new_token(320 + P, len(ctx), 16, 8)
    check_fused(kv, tok, num_partitions)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (24, 8), (32, 8), (64, 8), (4, 1)])
def test_fused_step_group_sizes(Hq, Hkv):
    ctx = [700, 33]
    kv = inputs.paged_kv(340 + Hq, ctx, Hkv=Hkv, page_size=16)
    tok = inputs.new_token(340 + Hq, len(ctx), Hq, Hkv)
    check_fused(kv, tok, 0)
    check_fused(kv, tok, 4)


@pytest.mark.parametrize("num_partitions", [0, 2, 70])
def test_fused_step_matches_the_two_launches_bit_for_bit(num_partitions):
    ctx = [5000, 129, 1]
    kv = inputs.paged_kv(360, ctx, Hkv=8, page_size=16)
    tok = inputs.new_token(360, len(ctx), 32, 8)
    fused = run_fused(kv, tok, num_partitions)
    two = run_unfused(kv, tok, num_partitions)
    for key in ("q_out", "kc", "vc", "ob"):
        assert np.array_equal(fused[key], two[key]), key
    assert np.array_equal(fused["of"], two["of"])


@pytest.mark.parametrize("Hq,ctx,num_partitions,P", [
    (8, [5000, 129, 1], 100, 16),   # g = 1 (79 partitions); a one-partition sequence writes its output
    (24, [3000, 40, 700], 100, 16), # g = 3 (94 partitions of 32 positions)
    (32, [6000, 16, 2047], 200, 16),  # one-page partitions: 4 of 6 warps own no chunk
    (16, [20000], 100, 16),         # one sequence: 19 CTAs per KV head
    (16, [20000, 333], 100, 64),    # 64-position pages: four chunks per page
])
def test_walked_partitions_equal_the_two_cta_shape(Hq, ctx, num_partitions, P):
    """Attention alone over these grids walks runs of partitions per CTA;
    the fused step keeps the two-CTA shape, one partition per CTA. Every
    partition is folded by the same warps in the same pairs and merged in
    the same order, so the two agree bit for bit, and both with the oracle."""
    kv = inputs.paged_kv(370 + Hq + len(ctx) + P, ctx, Hkv=8, page_size=P)
    assert walked(len(ctx), Hq, 8, P, kv.max_pages, num_partitions)
    tok = inputs.new_token(370 + Hq, len(ctx), Hq, 8)
    fused = check_fused(kv, tok, num_partitions)
    two = run_unfused(kv, tok, num_partitions)
    for key in ("q_out", "kc", "vc", "ob"):
        assert np.array_equal(fused[key], two[key]), key
    assert np.array_equal(fused["of"], two["of"])
    assert pg.device_error_flags() == 0


@pytest.mark.parametrize("Hq", [8, 24, 48])
def test_fused_step_two_cta_shape(Hq):
    # several waves of short partitions (8 sequences x 8 KV heads x 40
    # partitions of 64 positions) run the two-CTA shape, 6 warps: g = 1, 3
    # and 6 (as many query heads per KV head as it has warps to rotate them);
    # against the oracle and bit for bit against the two launches
    ctx = [2048, 1, 2, 1500, 2047, 700, 2048, 33]
    kv = inputs.paged_kv(380 + Hq, ctx, Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(380 + Hq, len(ctx), Hq, 8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    np_used = pg.decode_attn_partition_count(len(ctx), 8, 16, kv.max_pages, 40)
    assert np_used > 1 and len(ctx) * 8 * np_used > sms and -(-kv.max_pages // np_used) * 16 <= 2048
    fused = check_fused(kv, tok, 40)
    two = run_unfused(kv, tok, 40)
    for key in ("q_out", "kc", "vc", "ob"):
        assert np.array_equal(fused[key], two[key]), key
    assert np.array_equal(fused["of"], two["of"])


def test_fused_step_flags_empty_context_and_bad_page():
    kv = inputs.paged_kv(370, [40, 40], Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(370, 2, 16, 8)
    kv.context_lens[0] = 0
    kv.block_table[1, 2] = kv.num_pages + 9  # page of position 39
    got = run_fused(kv, tok, 0)
    flags = pg.device_error_flags()
    assert flags & binding.DEVERR_BAD_CONTEXT and flags & binding.DEVERR_BAD_PAGE
    assert np.all(got["of"][0] == 0)
    assert np.isfinite(got["of"]).all()
