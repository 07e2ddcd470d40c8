"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Bars (from the decode-attention spec): cache-append addressing and V copies
bit-exact; q_out and appended K within 1 bf16 ulp of the oracle's rounding;
attention outputs within 2e-3 absolute (fp32) and within 1 bf16 ulp of the
oracle's rounded result (bf16 output).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import inputs
from parity_util import assert_bf16_close, walked
from paged_gqa_decode_head_gb300.runner import DecodeStep, bf16_bits, to_device_bf16, to_device_i32

pytestmark = pytest.mark.gpu

ATOL_F32 = 2e-3
THETA = 1e6
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(autouse=True)
def _clean_flags():
    pg.device_error_flags(clear=True)
    yield


def gpu_decode(q_bits, kv, scale=SCALE, num_partitions=0, out_f32=True, out_bf16=True):
    dev = "cuda"
    q = to_device_bf16(q_bits, dev)
    kc = to_device_bf16(kv.k_cache, dev)
    vc = to_device_bf16(kv.v_cache, dev)
    bt = to_device_i32(kv.block_table, dev)
    ctx = to_device_i32(kv.context_lens, dev)
    B, Hq, D = q_bits.shape
    Hkv = kv.k_cache.shape[1]
    ws_bytes = pg.decode_attn_workspace_size(B, Hq, Hkv, D, kv.page_size, kv.max_pages, num_partitions)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    of = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev) if out_f32 else None
    ob = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev) if out_bf16 else None
    pg.decode_attn_paged(q, kc, vc, bt, ctx, scale, out_f32=of, out_bf16=ob, workspace=ws,
                         num_partitions=num_partitions)
    torch.cuda.synchronize()
    return (of.cpu().numpy() if of is not None else None), (bf16_bits(ob) if ob is not None else None)


def check_attention(q_bits, kv, num_partitions=0, scale=SCALE):
    ref = oracle.decode_attention(q_bits, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, scale)
    of, ob = gpu_decode(q_bits, kv, scale, num_partitions)
    err = np.abs(of.astype(np.float64) - ref)
    assert np.isfinite(of).all()
    assert err.max() <= ATOL_F32, f"max abs err {err.max():.3e} (NP={num_partitions})"
    assert_bf16_close(ob, oracle.round_bf16(ref))
    assert pg.device_error_flags() == 0
    return err.max()


# ------------------------------------------------------------------ prologue
def check_prologue(kv, tok, theta=THETA):
    B, Hq, D = tok.q.shape
    Hkv = tok.k.shape[1]
    dev = "cuda"
    kc = to_device_bf16(kv.k_cache, dev)
    vc = to_device_bf16(kv.v_cache, dev)
    q_out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append(to_device_bf16(tok.q, dev), to_device_bf16(tok.k, dev), to_device_bf16(tok.v, dev),
                           to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev),
                           to_device_i32(kv.context_lens, dev), to_device_i32(kv.block_table, dev), kc, vc, q_out,
                           kv.page_size, theta)
    torch.cuda.synchronize()
    q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                       kv.context_lens, kv.block_table, kv.k_cache, kv.v_cache,
                                                       kv.page_size, theta)
    kc_gpu, vc_gpu = bf16_bits(kc), bf16_bits(vc)
    assert_bf16_close(bf16_bits(q_out), q_ref)
    # slots: exactly the oracle's slots changed, V bit for bit, K within 1 ulp
    assert np.array_equal(vc_gpu, vc_ref)
    changed = np.any(kc_gpu != kv.k_cache, axis=-1) | np.any(kc_ref != kv.k_cache, axis=-1)
    untouched = ~changed
    assert np.array_equal(kc_gpu[untouched], kv.k_cache[untouched])
    assert_bf16_close(kc_gpu, kc_ref)
    assert pg.device_error_flags() == 0
    return bf16_bits(q_out), kc_gpu, vc_gpu


def test_prologue_tiny_workload():
    w = inputs.WORKLOADS["tiny_t512"]
    kv = inputs.paged_kv(w["seed"], [w["T"]], Hkv=w["Hkv"], page_size=w["page_size"], fill_unused="normal")
    tok = inputs.new_token(w["seed"], 1, w["Hq"], w["Hkv"])
    check_prologue(kv, tok)


@pytest.mark.parametrize("P", [16, 32, 256])
def test_prologue_ragged_positions(P):
    ctx = [1, 15, 16, 17, 300, 4097]
    kv = inputs.paged_kv(31, ctx, Hkv=8, page_size=P, fill_unused="nan")
    tok = inputs.new_token(31, len(ctx), 32, 8)
    check_prologue(kv, tok)


def test_prologue_large_positions_keep_rope_accuracy():
    ctx = [131072, 65536, 100003]
    kv = inputs.paged_kv(32, ctx, Hkv=2, page_size=256, fill_unused="normal")
    tok = inputs.new_token(32, len(ctx), 4, 2)
    check_prologue(kv, tok)


def test_prologue_rejects_bad_context_and_page_on_device():
    kv = inputs.paged_kv(33, [20, 20], Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(33, 2, 16, 8)
    kv.context_lens[0] = 0  # no new token position
    kv.block_table[1, 1] = kv.num_pages + 3  # page of position 19 outside the pool
    dev = "cuda"
    kc = to_device_bf16(kv.k_cache, dev)
    vc = to_device_bf16(kv.v_cache, dev)
    q_out = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append(to_device_bf16(tok.q, dev), to_device_bf16(tok.k, dev), to_device_bf16(tok.v, dev),
                           to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev),
                           to_device_i32(kv.context_lens, dev), to_device_i32(kv.block_table, dev), kc, vc, q_out,
                           16, THETA)
    flags = pg.device_error_flags()
    assert flags & binding_flag("BAD_CONTEXT") and flags & binding_flag("BAD_PAGE")
    assert np.array_equal(bf16_bits(kc), kv.k_cache)  # nothing written anywhere
    assert np.array_equal(bf16_bits(vc), kv.v_cache)


def binding_flag(name):
    from paged_gqa_decode_head_gb300 import binding

    return getattr(binding, "DEVERR_" + name)


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("T", list(range(1, 9)))
def test_decode_bruteforce_small_contexts(T):
    kv = inputs.paged_kv(40 + T, [T], Hkv=8, page_size=16)
    q = inputs.query(40 + T, 1, 16)
    check_attention(q, kv)


def test_decode_t1_returns_v_exactly():
    kv = inputs.paged_kv(49, [1, 1], Hkv=8, page_size=16)
    q = inputs.query(49, 2, 16)
    of, ob = gpu_decode(q, kv)
    for b in range(2):
        page = kv.block_table[b, 0]
        for h in range(16):
            v = inputs.bf16_bits_to_f32(kv.v_cache[page, h // 2, 0])
            assert np.array_equal(of[b, h], v)
            assert np.array_equal(ob[b, h], kv.v_cache[page, h // 2, 0])


@pytest.mark.parametrize("T", [15, 16, 17, 31, 32, 33, 511, 512, 513])
@pytest.mark.parametrize("num_partitions", [0, 1, 2])
def test_decode_page_boundaries(T, num_partitions):
    kv = inputs.paged_kv(50 + T, [T], Hkv=8, page_size=16)
    q = inputs.query(50 + T, 1, 16)
    check_attention(q, kv, num_partitions)


@pytest.mark.parametrize("num_partitions", [0, 1, 2, 3, 4, 8, 32])
def test_decode_tiny_workload_partitions(num_partitions):
    w = inputs.WORKLOADS["tiny_t512"]
    kv = inputs.paged_kv(w["seed"], [w["T"]], Hkv=w["Hkv"], page_size=w["page_size"])
    q = inputs.query(w["seed"], 1, w["Hq"])
    check_attention(q, kv, num_partitions)


@pytest.mark.parametrize("P", [16, 32, 64, 128, 256])
def test_decode_page_sizes(P):
    ctx = [1, P - 1, P, P + 1, 5 * P + 3, 700]
    kv = inputs.paged_kv(60 + P, ctx, Hkv=8, page_size=P)
    q = inputs.query(60 + P, len(ctx), 16)
    for np_ in (0, 1, 3):
        check_attention(q, kv, np_)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (24, 8), (32, 8), (40, 8), (48, 8), (56, 8), (64, 8), (4, 1)])
def test_decode_group_sizes(Hq, Hkv):
    ctx = [300, 17, 1029]
    kv = inputs.paged_kv(70 + Hq, ctx, Hkv=Hkv, page_size=16)
    q = inputs.query(70 + Hq, len(ctx), Hq)
    check_attention(q, kv, 0)
    check_attention(q, kv, 5)


@pytest.mark.parametrize("num_partitions", [65, 94, 188])
def test_decode_many_partitions_use_the_merge_kernel(num_partitions):
    # more partitions than the split kernel merges in its last CTA
    ctx = [3000, 1500, 40]
    kv = inputs.paged_kv(86, ctx, Hkv=8, page_size=16)
    q = inputs.query(86, len(ctx), 32)
    check_attention(q, kv, num_partitions)


def two_cta_shape(B, Hq, Hkv, P, max_pages, num_partitions):
    """The library's rule for its two-CTAs-per-SM kernel shape (6 warps x 2
    stages): one new token, g <= 6, more CTAs than SMs and partitions of at
    most 2048 positions."""
    np_used = pg.decode_attn_partition_count(B, Hkv, P, max_pages, num_partitions)
    ppp = -(-max_pages // np_used)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return Hq // Hkv <= 6 and np_used > 1 and ppp * P <= 2048 and B * Hkv * np_used > sms


@pytest.mark.parametrize("Hq,num_partitions", [(8, 64), (16, 32), (32, 24), (48, 40), (48, 8)])
def test_decode_two_cta_shape_in_kernel_and_kernel_merges(Hq, num_partitions):
    # several waves of short partitions run the two-CTA shape; (48, 40) has
    # more accumulators than its stage area holds and merges in merge_kernel,
    # the others in the last CTA; empty and one-position sequences included
    ctx = [2048, 1, 0, 1500, 2047, 700, 2048, 33]
    kv = inputs.paged_kv(95 + Hq, ctx, Hkv=8, page_size=16)
    q = inputs.query(95 + Hq, len(ctx), Hq)
    assert two_cta_shape(len(ctx), Hq, 8, 16, kv.max_pages, num_partitions)
    check_attention(q, kv, num_partitions)


def test_decode_two_cta_shape_is_taken_only_for_short_partitions_in_several_waves():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # the T = 8192 layer chain and a long single sequence fit one wave
    assert not two_cta_shape(1, 16, 8, 16, 512, 0)
    assert not two_cta_shape(1, 32, 8, 16, 8192, 0)
    # 512-position partitions of T = 131072: 2048 CTAs
    assert two_cta_shape(1, 32, 8, 16, 8192, 256)
    # 4096-position partitions stay on the one-CTA shape
    assert not two_cta_shape(1, 32, 8, 16, 8192, 32)
    # groups of 8 query heads need the one-CTA shape's 9 warps
    assert not two_cta_shape(1, 64, 8, 16, 8192, 256)
    assert 8 * 256 > sms


def test_decode_repeated_calls_reuse_the_workspace():
    # the partition tickets must come back to zero after every call
    kv = inputs.paged_kv(87, [2000, 3001], Hkv=8, page_size=16)
    q = inputs.query(87, 2, 16)
    dev = "cuda"
    args = (to_device_bf16(q, dev), to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev),
            to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev), SCALE)
    ws = torch.zeros(pg.decode_attn_workspace_size(2, 16, 8, 128, 16, kv.max_pages, 12), dtype=torch.uint8,
                     device=dev)
    outs = []
    for _ in range(3):
        out = torch.full((2, 16, 128), float("nan"), device=dev)
        pg.decode_attn_paged(*args, out_f32=out, workspace=ws, num_partitions=12)
        outs.append(out)
    torch.cuda.synchronize()
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
    for out in outs:
        assert np.abs(out.cpu().numpy() - ref).max() <= ATOL_F32
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_decode_ragged_batch_with_empty_sequence():
    ctx = [0, 1, 17, 100, 513, 1000, 4096, 33]
    kv = inputs.paged_kv(80, ctx, Hkv=8, page_size=16)
    q = inputs.query(80, len(ctx), 16)
    for np_ in (0, 1, 4, 64):
        check_attention(q, kv, np_)
    of, ob = gpu_decode(q, kv)
    assert np.all(of[0] == 0) and np.all(ob[0] == 0)


def test_decode_output_variants_agree():
    kv = inputs.paged_kv(81, [777, 5], Hkv=8, page_size=16)
    q = inputs.query(81, 2, 16)
    both_f, both_b = gpu_decode(q, kv, num_partitions=3)
    only_f, _ = gpu_decode(q, kv, num_partitions=3, out_bf16=False)
    _, only_b = gpu_decode(q, kv, num_partitions=3, out_f32=False)
    assert np.array_equal(both_f, only_f) and np.array_equal(both_b, only_b)


def test_decode_rescale_stress():
    T = 3000
    kv = inputs.paged_kv(82, [T], Hkv=8, page_size=16)
    inputs.scale_key_outliers(kv, 82, fraction=0.01, factor=8.0)
    q = inputs.query(82, 1, 32)
    for np_ in (0, 1, 6):
        check_attention(q, kv, np_)


def test_decode_bad_page_and_context_are_masked_and_flagged():
    ctx = [64, 64]
    kv = inputs.paged_kv(83, ctx, Hkv=8, page_size=16, fill_unused="normal")
    q = inputs.query(83, 2, 16)
    kv.block_table[0, 2] = -7  # positions 32..47 of sequence 0 unreadable
    of, _ = gpu_decode(q, kv, num_partitions=2)
    flags = pg.device_error_flags()
    assert flags & binding_flag("BAD_PAGE")
    assert np.isfinite(of).all()
    # sequence 1 is unaffected
    good = inputs.PagedKV(kv.k_cache, kv.v_cache, kv.block_table[1:].copy(), kv.context_lens[1:].copy(), 16)
    ref = oracle.decode_attention(q[1:], good.k_cache, good.v_cache, good.block_table, good.context_lens, SCALE)
    assert np.abs(of[1:] - ref).max() <= ATOL_F32
    # a context longer than the table allows
    kv2 = inputs.paged_kv(84, [32], Hkv=8, page_size=16, fill_unused="normal")
    kv2.context_lens[0] = 10_000
    of, _ = gpu_decode(q[:1], kv2)
    assert pg.device_error_flags() & binding_flag("BAD_CONTEXT")
    assert np.all(of == 0)


def test_walked_partitions_mask_and_flag_bad_pages_and_contexts():
    """The same rules on a walked grid (runs of partitions per CTA): a refused
    page is masked and flagged, a context longer than the table gives zeros
    and a flag, the other sequences are unaffected."""
    ctx = [3000, 2500, 1000]
    kv = inputs.paged_kv(87, ctx, Hkv=8, page_size=16, fill_unused="normal")
    q = inputs.query(87, len(ctx), 16)
    assert walked(len(ctx), 16, 8, 16, kv.max_pages, 100)
    kv.block_table[0, 40] = -3          # positions 640..655 of sequence 0 unreadable
    kv.context_lens[2] = kv.max_pages * 16 + 1
    of, _ = gpu_decode(q, kv, num_partitions=100)
    flags = pg.device_error_flags()
    assert flags & binding_flag("BAD_PAGE") and flags & binding_flag("BAD_CONTEXT")
    assert np.isfinite(of).all()
    assert np.all(of[2] == 0)
    good = inputs.PagedKV(kv.k_cache, kv.v_cache, kv.block_table[1:2].copy(), kv.context_lens[1:2].copy(), 16)
    ref = oracle.decode_attention(q[1:2], good.k_cache, good.v_cache, good.block_table, good.context_lens, SCALE)
    assert np.abs(of[1:2] - ref).max() <= ATOL_F32


def test_decode_workspace_too_small_is_refused():
    kv = inputs.paged_kv(85, [1000], Hkv=8, page_size=16)
    dev = "cuda"
    q = to_device_bf16(inputs.query(85, 1, 16), dev)
    out = torch.empty((1, 16, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(64, dtype=torch.uint8, device=dev)
    with pytest.raises(pg.PgqaError) as e:
        pg.decode_attn_paged(q, to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev),
                             to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev), SCALE,
                             out_f32=out, workspace=ws, num_partitions=4)
    assert e.value.status == -4


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("NP", [1, 2, 5, 256, 1000])
def test_partition_merge_matches_oracle(NP):
    gen = np.random.default_rng(NP)
    B, Hq, D = 2, 4, 128
    m = (gen.standard_normal((B, Hq, NP)) * 5).astype(np.float32)
    l = gen.uniform(0.5, 50.0, (B, Hq, NP)).astype(np.float32)
    acc = gen.standard_normal((B, Hq, NP, D)).astype(np.float32)
    if NP > 1:  # some empty partitions
        empty = gen.random((B, Hq, NP)) < 0.3
        empty[..., 0] = False
        m[empty], l[empty] = -1e30, 0.0
        acc[empty] = 0.0
    dev = "cuda"
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    outb = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    pg.attn_partition_merge(torch.from_numpy(m).to(dev), torch.from_numpy(l).to(dev), torch.from_numpy(acc).to(dev),
                            out_f32=out, out_bf16=outb)
    torch.cuda.synchronize()
    ref = oracle.merge_partitions_batched(m, l, acc)
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())
    assert_bf16_close(bf16_bits(outb), oracle.round_bf16(ref))


def test_partition_merge_all_empty_is_zero():
    dev = "cuda"
    m = torch.full((1, 2, 3), -1e30, device=dev)
    l = torch.zeros((1, 2, 3), device=dev)
    acc = torch.zeros((1, 2, 3, 128), device=dev)
    out = torch.full((1, 2, 128), 7.0, device=dev)
    pg.attn_partition_merge(m, l, acc, out_f32=out)
    assert torch.all(out == 0)


# ------------------------------------------------------------------ host-tiled
def _tile_state_gpu(q, k, v, tile):
    dev = "cuda"
    B, Hq, D = q.shape
    _, T, Hkv, _ = k.shape
    qd = to_device_bf16(q, dev)
    m = torch.empty((B, Hq), device=dev)
    l = torch.empty((B, Hq), device=dev)
    acc = torch.empty((B, Hq, D), device=dev)
    pg.attn_tile_init(m, l, acc)
    kd = to_device_bf16(k, dev)
    vd = to_device_bf16(v, dev)
    for t0 in range(0, T, tile):
        n = min(tile, T - t0)
        kt = kd[:, t0:t0 + n].contiguous()
        vt = vd[:, t0:t0 + n].contiguous()
        pg.attn_tile_update(qd, kt, vt, m, l, acc, SCALE)
    return m, l, acc


@pytest.mark.parametrize("B,T,Hq,Hkv", [(1, 2000, 16, 8), (2, 513, 32, 8), (1, 16, 8, 8)])
def test_tile_update_state_and_output(B, T, Hq, Hkv):
    k, v = inputs.contiguous_kv(90 + T, B, T, Hkv)
    q = inputs.query(90 + T, B, Hq)
    m, l, acc = _tile_state_gpu(q, k, v, 512)
    out = torch.empty((B, Hq, 128), device="cuda")
    outb = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    pg.attn_tile_finalize(m, l, acc, out_f32=out, out_bf16=outb)
    torch.cuda.synchronize()
    ref = oracle.attention_contiguous(q, k, v, SCALE)
    assert np.abs(out.cpu().numpy() - ref).max() <= ATOL_F32
    assert_bf16_close(bf16_bits(outb), oracle.round_bf16(ref))
    # the state itself: m is the running max; l and acc relative to it
    m_ref, l_ref, acc_ref = oracle.tiled_state_reference(q, k, v, SCALE, 512)
    mg, lg, ag = m.cpu().numpy(), l.cpu().numpy(), acc.cpu().numpy()
    assert np.abs(mg - m_ref).max() <= 1e-4 * max(1.0, np.abs(m_ref).max())
    assert np.abs(lg / l_ref - 1).max() <= 1e-3
    assert np.abs(ag / lg[..., None] - acc_ref / l_ref[..., None]).max() <= ATOL_F32


def test_tile_state_resumes_like_a_checkpoint():
    # finalize after the first tiles, keep going, finalize again: each result
    # equals direct attention over the prefix seen so far
    B, T, Hq, Hkv = 1, 1536, 16, 8
    k, v = inputs.contiguous_kv(95, B, T, Hkv)
    q = inputs.query(95, B, Hq)
    dev = "cuda"
    qd, kd, vd = to_device_bf16(q, dev), to_device_bf16(k, dev), to_device_bf16(v, dev)
    m = torch.empty((B, Hq), device=dev)
    l = torch.empty((B, Hq), device=dev)
    acc = torch.empty((B, Hq, 128), device=dev)
    pg.attn_tile_init(m, l, acc)
    out = torch.empty((B, Hq, 128), device=dev)
    for t0 in range(0, T, 512):
        pg.attn_tile_update(qd, kd[:, t0:t0 + 512].contiguous(), vd[:, t0:t0 + 512].contiguous(), m, l, acc, SCALE)
        pg.attn_tile_finalize(m, l, acc, out_f32=out)
        torch.cuda.synchronize()
        ref = oracle.attention_contiguous(q, np.ascontiguousarray(k[:, :t0 + 512]),
                                          np.ascontiguousarray(v[:, :t0 + 512]), SCALE)
        assert np.abs(out.cpu().numpy() - ref).max() <= ATOL_F32


def host_tiled(q, k, v, tile=512, n_slots=2, tiles_per_copy=1, trace_events=None):
    dev = "cuda"
    B, Hq, D = q.shape
    _, T, Hkv, _ = k.shape
    hk = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
    span = tile * tiles_per_copy
    slots_k = [torch.full((B, span, Hkv, D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(n_slots)]
    slots_v = [torch.full((B, span, Hkv, D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(n_slots)]
    events = [torch.cuda.Event() for _ in range(2 * n_slots)]
    m = torch.empty((B, Hq), device=dev)
    l = torch.empty((B, Hq), device=dev)
    acc = torch.empty((B, Hq, D), device=dev)
    out = torch.empty((B, Hq, D), device=dev)
    outb = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    copy_stream = torch.cuda.Stream()
    pg.attn_host_tiled_run(to_device_bf16(q, dev), hk, hv, SCALE, slots_k, slots_v, events, m, l, acc,
                           out_f32=out, out_bf16=outb, tile_len=tile, tiles_per_copy=tiles_per_copy,
                           copy_stream=copy_stream, trace_events=trace_events)
    torch.cuda.synchronize()
    return out.cpu().numpy(), bf16_bits(outb)


@pytest.mark.parametrize("per_copy", [1, 4])
def test_host_tiled_run_traced_gives_the_same_bits_and_ordered_events(per_copy):
    """The traced pipeline computes exactly what the plain one does; its
    events, per copy group, come in the order copy start <= copy end <=
    update start <= update end, and a group's update starts after its copy."""
    T, tile = 3000, 512
    k, v = inputs.contiguous_kv(97, 1, T, 8)
    q = inputs.query(97, 1, 16)
    plain = host_tiled(q, k, v, tile, 2, per_copy)
    groups = -(-T // (tile * per_copy))
    trace = [torch.cuda.Event(enable_timing=True) for _ in range(4 * groups)]
    traced = host_tiled(q, k, v, tile, 2, per_copy, trace_events=trace)
    assert np.array_equal(plain[0], traced[0]) and np.array_equal(plain[1], traced[1])
    t = [trace[0].elapsed_time(ev) for ev in trace]
    for g in range(groups):
        c0, c1, u0, u1 = t[4 * g:4 * g + 4]
        assert 0.0 <= c0 <= c1 <= u0 <= u1


@pytest.mark.parametrize("B,T,tile,n_slots,per_copy", [
    (1, 4096, 512, 2, 1), (2, 1500, 512, 3, 1), (1, 700, 128, 2, 1), (3, 1, 512, 2, 1),
    (1, 4096, 512, 2, 4), (2, 5000, 512, 2, 3), (3, 1300, 128, 3, 2), (1, 100, 512, 2, 8)])
def test_host_tiled_run_matches_oracle(B, T, tile, n_slots, per_copy):
    """Copies of one tile (the pages' pipeline) or of several tiles per slot
    (per_copy), ragged last groups and tiles, several sequences."""
    k, v = inputs.contiguous_kv(96 + T, B, T, 8)
    q = inputs.query(96 + T, B, 16)
    out, outb = host_tiled(q, k, v, tile, n_slots, per_copy)
    ref = oracle.attention_contiguous(q, k, v, SCALE)
    assert np.abs(out - ref).max() <= ATOL_F32
    assert_bf16_close(outb, oracle.round_bf16(ref))


# ------------------------------------------------------------------ composed step
def test_step_chain_prologue_then_attention_and_graph_replay():
    """p1's lesson: units can pass while the composition fails, so check the
    whole chain (prologue -> cache -> attention) over several layers, eager and
    as one CUDA graph."""
    layers = []
    for i in range(3):
        kv = inputs.paged_kv(100 + i, [257, 40], Hkv=8, page_size=16, fill_unused="nan")
        tok = inputs.new_token(100 + i, 2, 16, 8)
        layers.append((kv, tok))
    step = DecodeStep(layers, Hq=16, Hkv=8, rope_theta=THETA, num_partitions=2)
    step.run()
    torch.cuda.synchronize()
    eager = [st.out_f32.clone() for st in step.layers]
    for (kv, tok), st in zip(layers, step.layers):
        q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                           kv.context_lens, kv.block_table, kv.k_cache, kv.v_cache,
                                                           16, THETA)
        ref = oracle.decode_attention(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
        assert np.abs(st.out_f32.cpu().numpy() - ref).max() <= ATOL_F32
    step.capture()
    for st in step.layers:
        st.out_f32.zero_()
    step.replay()
    torch.cuda.synchronize()
    for a, st in zip(eager, step.layers):
        assert torch.equal(a, st.out_f32)
    assert pg.device_error_flags() == 0


def test_step_graph_with_host_io():
    """A step graph that starts with the copy of the new tokens from pinned
    host memory and ends with the copy of the outputs back: its host results
    equal the outputs of the same step run eagerly from device inputs."""
    layers = []
    for i in range(2):
        kv = inputs.paged_kv(110 + i, [300, 17], Hkv=8, page_size=16, fill_unused="normal")
        layers.append((kv, inputs.new_token(110 + i, 2, 16, 8)))
    eager = DecodeStep(layers, Hq=16, Hkv=8, rope_theta=THETA)
    eager.run(fused=True)
    torch.cuda.synchronize()
    step = DecodeStep(layers, Hq=16, Hkv=8, rope_theta=THETA)
    host_in = step.new_tokens.cpu().pin_memory()
    host_out = torch.full(step.outputs.shape, float("nan"), dtype=torch.float32).pin_memory()
    step.new_tokens.zero_()
    g = step.capture(fused=True, host_in=host_in, host_out=host_out)
    # the warm-up run before the capture already appended the new rows; the
    # replay appends them again (same slots, same values) and recomputes
    host_out.fill_(float("nan"))
    step.new_tokens.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(host_out, eager.outputs.cpu())
    assert torch.equal(step.new_tokens.cpu().view(torch.int16), host_in.view(torch.int16))
    with pytest.raises(ValueError):
        step.capture(host_in=host_in.to(torch.float32).pin_memory())
    assert pg.device_error_flags() == 0


def test_partition_count_follows_the_regime():
    """Automatic partition counts on this GPU: a T = 8192 layer of one
    sequence (latency-bound, every partition inside one CTA's ring) leaves at
    least a tenth of the SMs free; T = 131072 fills a wave of SMs; a batch
    that fills the SMs with its (sequence, KV head) units uses few
    partitions (16 sequences of 8192 positions: one each)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    short = pg.decode_attn_partition_count(1, 8, 16, 512, 0)
    assert 8 * short <= sms * 9 // 10 and short >= 2
    long_ = pg.decode_attn_partition_count(1, 8, 16, 8192, 0)
    assert sms * 9 // 10 < 8 * long_ <= sms
    assert pg.decode_attn_partition_count(16, 8, 16, 512, 0) == 1
