"""GPU parity of multi-query decode (M new tokens per sequence, token i at
position T - M + i attending causally): qk_norm_rope_append_multi and
decode_attn_paged_multi against the oracle's definitions."""
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

ATOL_F32 = 2e-3
SCALE = 1.0 / math.sqrt(128)
THETA = 1e6


@pytest.fixture(autouse=True)
def _clean_flags():
    pg.device_error_flags(clear=True)
    yield


def _queries(seed, B, M, Hq):
    return inputs.normal_bf16(inputs.generator(seed, 93), (B, M, Hq, 128))


def run_multi_attention(kv, q, num_partitions=0):
    B, M, Hq, _ = q.shape
    Hkv = kv.k_cache.shape[1]
    n = pg.decode_attn_multi_workspace_size(B, M, Hq, Hkv, 128, kv.page_size, kv.max_pages, num_partitions)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    of = torch.full((B, M, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.full((B, M, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pg.decode_attn_paged_multi(to_device_bf16(q, "cuda"), to_device_bf16(kv.k_cache, "cuda"),
                               to_device_bf16(kv.v_cache, "cuda"), to_device_i32(kv.block_table, "cuda"),
                               to_device_i32(kv.context_lens, "cuda"), SCALE, out_f32=of, out_bf16=ob, workspace=ws,
                               num_partitions=num_partitions)
    torch.cuda.synchronize()
    return of.cpu().numpy(), bf16_bits(ob)


def check_attention(kv, q, num_partitions=0):
    of, ob = run_multi_attention(kv, q, num_partitions)
    ref = oracle.decode_attention_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
    assert np.isfinite(of).all()
    assert np.abs(of - ref).max() <= ATOL_F32
    assert_bf16_close(ob, oracle.round_bf16(ref), "out_bf16")
    assert pg.device_error_flags() == 0
    return of


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [4, 5, 15, 16, 17, 18, 33, 700])
def test_multi_attention_small_contexts(M, T):
    kv = inputs.paged_kv(800 + 10 * M + T, [T, T + 1], Hkv=8, page_size=16)
    check_attention(kv, _queries(800 + T, 2, M, 16))


@pytest.mark.parametrize("num_partitions", [0, 1, 3, 70])
def test_multi_attention_partitions_and_ragged(num_partitions):
    ctx = [4, 17, 300, 4097, 2000]
    kv = inputs.paged_kv(850 + num_partitions, ctx, Hkv=8, page_size=16)
    check_attention(kv, _queries(850, len(ctx), 4, 16), num_partitions)


@pytest.mark.parametrize("Hq,Hkv,M", [(8, 8, 8), (8, 8, 5), (32, 8, 2), (24, 8, 2), (64, 8, 1), (4, 1, 2)])
def test_multi_attention_group_sizes(Hq, Hkv, M):
    kv = inputs.paged_kv(870 + Hq + M, [700, 33], Hkv=Hkv, page_size=16)
    check_attention(kv, _queries(870 + Hq, 2, M, Hq), 0)
    check_attention(kv, _queries(871 + Hq, 2, M, Hq), 5)


@pytest.mark.parametrize("P", [32, 256])
def test_multi_attention_page_sizes(P):
    kv = inputs.paged_kv(880 + P, [1000, 3 * P + 2], Hkv=8, page_size=P)
    check_attention(kv, _queries(880 + P, 2, 3, 16), 0)


def test_multi_attention_with_one_token_matches_decode_attn_paged_bit_for_bit():
    kv = inputs.paged_kv(890, [5000, 129, 1], Hkv=8, page_size=16)
    q = _queries(890, 3, 1, 16)
    of, ob = run_multi_attention(kv, q, 4)
    n = pg.decode_attn_workspace_size(3, 16, 8, 128, 16, kv.max_pages, 4)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    of1 = torch.empty((3, 16, 128), dtype=torch.float32, device="cuda")
    pg.decode_attn_paged(to_device_bf16(q[:, 0], "cuda"), to_device_bf16(kv.k_cache, "cuda"),
                         to_device_bf16(kv.v_cache, "cuda"), to_device_i32(kv.block_table, "cuda"),
                         to_device_i32(kv.context_lens, "cuda"), SCALE, out_f32=of1, workspace=ws, num_partitions=4)
    torch.cuda.synchronize()
    assert np.array_equal(of[:, 0], of1.cpu().numpy())


def test_multi_prologue_then_attention_chain():
    """qk_norm_rope_append_multi then decode_attn_paged_multi on its q_out, as
    a speculative-verification step does, against the oracle's chain."""
    M, ctx = 3, [40, 17, 600]
    B = len(ctx)
    kv = inputs.paged_kv(900, ctx, Hkv=8, page_size=16)
    g = inputs.generator(900, 94)
    q = inputs.normal_bf16(g, (B, M, 16, 128))
    k = inputs.normal_bf16(g, (B, M, 8, 128))
    v = inputs.normal_bf16(g, (B, M, 8, 128))
    tok = inputs.new_token(900, B, 16, 8)
    dev = "cuda"
    kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
    bt, cl = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
    q_out = torch.empty((B, M, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append_multi(to_device_bf16(q, dev), to_device_bf16(k, dev), to_device_bf16(v, dev),
                                 to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev), cl, bt, kc, vc,
                                 q_out, THETA)
    n = pg.decode_attn_multi_workspace_size(B, M, 16, 8, 128, 16, kv.max_pages, 0)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    of = torch.empty((B, M, 16, 128), dtype=torch.float32, device=dev)
    pg.decode_attn_paged_multi(q_out, kc, vc, bt, cl, SCALE, out_f32=of, workspace=ws)
    torch.cuda.synchronize()
    q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append_multi(q, k, v, tok.gamma_q, tok.gamma_k, kv.context_lens,
                                                             kv.block_table, kv.k_cache, kv.v_cache, 16, THETA)
    assert_bf16_close(bf16_bits(q_out), q_ref, "q_out")
    assert np.array_equal(bf16_bits(vc), vc_ref)
    kc_got = bf16_bits(kc)
    changed = np.any(kc_got != kv.k_cache, axis=-1) | np.any(kc_ref != kv.k_cache, axis=-1)
    assert np.array_equal(kc_got[~changed], kv.k_cache[~changed])
    assert_bf16_close(kc_got, kc_ref, "appended K")
    ref = oracle.decode_attention_multi(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
    assert np.abs(of.cpu().numpy() - ref).max() <= ATOL_F32
    assert pg.device_error_flags() == 0


def test_multi_refuses_too_many_columns_and_flags_short_contexts():
    kv = inputs.paged_kv(910, [2, 40], Hkv=8, page_size=16, fill_unused="normal")
    with pytest.raises(binding.PgqaError):
        run_multi_attention(kv, _queries(910, 2, 5, 16))  # 5 tokens x 2 heads > 8 columns
    of, _ = run_multi_attention(kv, _queries(911, 2, 3, 16))  # T = 2 < M = 3 for sequence 0
    assert pg.device_error_flags() & binding.DEVERR_BAD_CONTEXT
    assert np.all(of[0] == 0)
    assert np.isfinite(of).all()


def test_multi_short_context_with_the_separate_merge_kernel():
    """T < M with more than 64 partitions (the merge runs as its own kernel):
    the short sequence still gets zeros and the flag, the other its
    attention."""
    kv = inputs.paged_kv(912, [2, 2240], Hkv=8, page_size=16, fill_unused="normal")
    assert pg.decode_attn_partition_count(2, 8, 16, kv.max_pages, 70) > 64
    q = _queries(913, 2, 3, 16)
    of, _ = run_multi_attention(kv, q, num_partitions=70)
    assert pg.device_error_flags() & binding.DEVERR_BAD_CONTEXT
    assert np.all(of[0] == 0)
    ref = oracle.decode_attention_multi(q[1:], kv.k_cache, kv.v_cache, kv.block_table[1:], kv.context_lens[1:], SCALE)
    assert np.abs(of[1:] - ref).max() <= ATOL_F32


def test_multi_token_workload_layers_full_size():
    """Two layers of the multi-token verification workload (T = 8192, M = 4)
    at full size, prologue then attention, against the oracle's chain."""
    w = inputs.WORKLOADS["qwen3_0p6b_t8k_m4"]
    dev = "cuda"
    for kv, q, k, v, gq, gk in inputs.qwen3_layers_multi(layers=2):
        B, M = w["B"], w["M"]
        kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
        bt, cl = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
        q_out = torch.empty((B, M, w["Hq"], 128), dtype=torch.bfloat16, device=dev)
        pg.qk_norm_rope_append_multi(to_device_bf16(q, dev), to_device_bf16(k, dev), to_device_bf16(v, dev),
                                     to_device_bf16(gq, dev), to_device_bf16(gk, dev), cl, bt, kc, vc, q_out,
                                     w["theta"])
        n = pg.decode_attn_multi_workspace_size(B, M, w["Hq"], w["Hkv"], 128, kv.page_size, kv.max_pages, 0)
        ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
        of = torch.empty((B, M, w["Hq"], 128), dtype=torch.float32, device=dev)
        pg.decode_attn_paged_multi(q_out, kc, vc, bt, cl, SCALE, out_f32=of, workspace=ws)
        torch.cuda.synchronize()
        q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append_multi(q, k, v, gq, gk, kv.context_lens, kv.block_table,
                                                                 kv.k_cache, kv.v_cache, kv.page_size, w["theta"])
        assert_bf16_close(bf16_bits(q_out), q_ref, "q_out")
        ref = oracle.decode_attention_multi(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
        assert np.abs(of.cpu().numpy() - ref).max() <= ATOL_F32
    assert pg.device_error_flags() == 0


def _fused_multi_case(seed, ctx, M, Hq=16, Hkv=8, P=16):
    B = len(ctx)
    kv = inputs.paged_kv(seed, ctx, Hkv=Hkv, page_size=P)
    g = inputs.generator(seed, 95)
    q = inputs.normal_bf16(g, (B, M, Hq, 128))
    k = inputs.normal_bf16(g, (B, M, Hkv, 128))
    v = inputs.normal_bf16(g, (B, M, Hkv, 128))
    tok = inputs.new_token(seed, B, Hq, Hkv)
    return kv, q, k, v, tok


def run_fused_multi(kv, q, k, v, tok, num_partitions=0):
    dev = "cuda"
    B, M, Hq, _ = q.shape
    Hkv = k.shape[2]
    kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
    q_out = torch.full((B, M, Hq, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    of = torch.full((B, M, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    ob = torch.full((B, M, Hq, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    n = pg.decode_attn_multi_workspace_size(B, M, Hq, Hkv, 128, kv.page_size, kv.max_pages, num_partitions)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    pg.decode_step_paged_multi(to_device_bf16(q, dev), to_device_bf16(k, dev), to_device_bf16(v, dev),
                               to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev),
                               to_device_i32(kv.context_lens, dev), to_device_i32(kv.block_table, dev), kc, vc, SCALE,
                               THETA, q_out=q_out, out_f32=of, out_bf16=ob, workspace=ws,
                               num_partitions=num_partitions)
    torch.cuda.synchronize()
    return dict(q_out=bf16_bits(q_out), kc=bf16_bits(kc), vc=bf16_bits(vc), of=of.cpu().numpy(), ob=bf16_bits(ob))


def check_fused_multi(kv, q, k, v, tok, num_partitions=0):
    got = run_fused_multi(kv, q, k, v, tok, num_partitions)
    q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append_multi(q, k, v, tok.gamma_q, tok.gamma_k, kv.context_lens,
                                                             kv.block_table, kv.k_cache, kv.v_cache, kv.page_size,
                                                             THETA)
    assert_bf16_close(got["q_out"], q_ref, "q_out")
    assert np.array_equal(got["vc"], vc_ref)
    changed = np.any(got["kc"] != kv.k_cache, axis=-1) | np.any(kc_ref != kv.k_cache, axis=-1)
    assert np.array_equal(got["kc"][~changed], kv.k_cache[~changed])
    assert_bf16_close(got["kc"], kc_ref, "appended K")
    # the whole chain against the oracle's chain (fp32 bar); the attention
    # alone on the step's own q_out and cache (which may differ from the
    # oracle's by 1 bf16 ulp, checked above) for the bf16 bar
    ref = oracle.decode_attention_multi(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
    assert np.isfinite(got["of"]).all()
    assert np.abs(got["of"] - ref).max() <= ATOL_F32
    own = oracle.decode_attention_multi(got["q_out"], got["kc"], got["vc"], kv.block_table, kv.context_lens, SCALE)
    assert np.abs(got["of"] - own).max() <= ATOL_F32
    assert_bf16_close(got["ob"], oracle.round_bf16(own), "out_bf16")
    assert pg.device_error_flags() == 0
    return got


@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("T", [4, 15, 16, 17, 18, 19, 20, 33, 513])
def test_fused_multi_step_small_contexts(M, T):
    """New tokens inside one chunk, straddling a chunk or page boundary."""
    check_fused_multi(*_fused_multi_case(920 + 10 * M + T, [T, T + 3], M))


@pytest.mark.parametrize("num_partitions", [0, 1, 3, 70])
def test_fused_multi_step_partitions(num_partitions):
    """Including new tokens split across two partitions (NP = 70: 1 page each)."""
    ctx = [4, 18, 300, 4097, 2002]
    check_fused_multi(*_fused_multi_case(950 + num_partitions, ctx, 4), num_partitions)


@pytest.mark.parametrize("Hq,Hkv,M", [(8, 8, 8), (32, 8, 2), (24, 8, 2), (4, 1, 2)])
def test_fused_multi_step_group_sizes(Hq, Hkv, M):
    check_fused_multi(*_fused_multi_case(960 + Hq + M, [700, 35], M, Hq, Hkv), 0)
    check_fused_multi(*_fused_multi_case(961 + Hq + M, [700, 35], M, Hq, Hkv), 5)


def test_fused_multi_step_matches_the_two_launches():
    kv, q, k, v, tok = _fused_multi_case(970, [5000, 129, 7], 3)
    fused = run_fused_multi(kv, q, k, v, tok, 4)
    dev = "cuda"
    kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
    bt, cl = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
    q_out = torch.empty((3, 3, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append_multi(to_device_bf16(q, dev), to_device_bf16(k, dev), to_device_bf16(v, dev),
                                 to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev), cl, bt, kc, vc,
                                 q_out, THETA)
    n = pg.decode_attn_multi_workspace_size(3, 3, 16, 8, 128, 16, kv.max_pages, 4)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    of = torch.empty((3, 3, 16, 128), dtype=torch.float32, device=dev)
    pg.decode_attn_paged_multi(q_out, kc, vc, bt, cl, SCALE, out_f32=of, workspace=ws, num_partitions=4)
    torch.cuda.synchronize()
    assert np.array_equal(fused["q_out"], bf16_bits(q_out))
    assert np.array_equal(fused["kc"], bf16_bits(kc)) and np.array_equal(fused["vc"], bf16_bits(vc))
    assert np.array_equal(fused["of"], of.cpu().numpy())
