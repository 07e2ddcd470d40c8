"""GPU parity of the INT8 KV cache: qk_norm_rope_append_int8 and
decode_attn_paged_int8 against the oracle's INT8 definitions, and a quality
gate of INT8 attention against bf16 attention on the same history."""
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


def int8_cache(kv):
    """The oracle's INT8 quantization of a bf16 paged cache; scales of slots
    past each sequence's end are set to NaN (the kernel must never use them)."""
    k8, ks = oracle.quantize_rows_int8(kv.k_cache)
    v8, vs = oracle.quantize_rows_int8(kv.v_cache)
    P = kv.page_size
    for b, T in enumerate(kv.context_lens):
        if T % P:
            page = kv.block_table[b, T // P]
            if 0 <= page < kv.num_pages:
                ks[page, :, T % P:] = np.nan
                vs[page, :, T % P:] = np.nan
    return k8, v8, ks, vs


def dev_i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).cuda()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def run_attention(kv, q, k8, v8, ks, vs, num_partitions=0):
    B, Hq, _ = q.shape
    Hkv = kv.k_cache.shape[1]
    n = pg.decode_attn_int8_workspace_size(B, Hq, Hkv, 128, kv.page_size, kv.max_pages, num_partitions)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    of = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pg.decode_attn_paged_int8(to_device_bf16(q, "cuda"), dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs),
                              to_device_i32(kv.block_table, "cuda"), to_device_i32(kv.context_lens, "cuda"), SCALE,
                              out_f32=of, out_bf16=ob, workspace=ws, num_partitions=num_partitions)
    torch.cuda.synchronize()
    return of.cpu().numpy(), bf16_bits(ob)


def check_attention(kv, q, num_partitions=0):
    k8, v8, ks, vs = int8_cache(kv)
    of, ob = run_attention(kv, q, k8, v8, ks, vs, num_partitions)
    ref = oracle.decode_attention_int8(q, k8, v8, ks, vs, kv.block_table, kv.context_lens, SCALE)
    assert np.isfinite(of).all()
    assert np.abs(of - ref).max() <= ATOL_F32
    assert_bf16_close(ob, oracle.round_bf16(ref), "out_bf16")
    assert pg.device_error_flags() == 0
    return of


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 33, 513, 1000])
def test_int8_attention_small_contexts(T):
    kv = inputs.paged_kv(1100 + T, [T, T + 5], Hkv=8, page_size=16, fill_unused="normal")
    check_attention(kv, inputs.query(1100 + T, 2, 16))


@pytest.mark.parametrize("num_partitions", [0, 1, 3, 70])
def test_int8_attention_ragged_and_partitions(num_partitions):
    ctx = [1, 17, 300, 4097, 2000]
    kv = inputs.paged_kv(1120 + num_partitions, ctx, Hkv=8, page_size=16, fill_unused="normal")
    check_attention(kv, inputs.query(1120, len(ctx), 16), num_partitions)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (24, 8), (32, 8), (64, 8), (4, 1)])
def test_int8_attention_group_sizes(Hq, Hkv):
    kv = inputs.paged_kv(1140 + Hq, [700, 33], Hkv=Hkv, page_size=16, fill_unused="normal")
    check_attention(kv, inputs.query(1140 + Hq, 2, Hq), 0)
    check_attention(kv, inputs.query(1141 + Hq, 2, Hq), 5)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (24, 8), (64, 8), (4, 1)])
@pytest.mark.parametrize("num_partitions", [1, 2])
def test_int8_attention_long_partitions(Hq, Hkv, num_partitions):
    """Partitions of 64 chunks (1024 positions) or more run the 16-warp CTA
    shape; a ragged tail and every group size on it."""
    kv = inputs.paged_kv(1150 + Hq + num_partitions, [2000, 1100, 7], Hkv=Hkv, page_size=16, fill_unused="normal")
    check_attention(kv, inputs.query(1150 + Hq, 3, Hq), num_partitions)


@pytest.mark.parametrize("Hq,num_partitions", [(16, 19), (8, 64), (16, 64), (64, 60)])
def test_int8_merge_paths_and_workspace_reuse(Hq, num_partitions):
    """Up to 64 partitions whose states fit the stage area are merged by the
    last CTA: these grids run four CTAs per SM (48 KiB of stages each), which
    hold 2 heads' states at 19 partitions and 1 head's at 64. 2 heads at 64
    and 8 at 60 do not fit and go to the merge kernel. The same workspace
    serves repeated calls (the ticket is left at zero) with identical
    results."""
    ctx = [3000, 64 * 16 + 3, 40]
    kv = inputs.paged_kv(1210 + num_partitions, ctx, Hkv=8, page_size=16, fill_unused="normal")
    q = inputs.query(1210 + num_partitions, len(ctx), Hq)
    k8, v8, ks, vs = int8_cache(kv)
    B = len(ctx)
    n = pg.decode_attn_int8_workspace_size(B, Hq, 8, 128, kv.page_size, kv.max_pages, num_partitions)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    args = (to_device_bf16(q, "cuda"), dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs),
            to_device_i32(kv.block_table, "cuda"), to_device_i32(kv.context_lens, "cuda"), SCALE)
    outs = []
    for _ in range(3):
        of = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        pg.decode_attn_paged_int8(*args, out_f32=of, workspace=ws, num_partitions=num_partitions)
        outs.append(of.cpu().numpy())
    ref = oracle.decode_attention_int8(q, k8, v8, ks, vs, kv.block_table, kv.context_lens, SCALE)
    assert np.abs(outs[0] - ref).max() <= ATOL_F32
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert pg.device_error_flags() == 0


@pytest.mark.parametrize("P", [32, 256])
def test_int8_attention_page_sizes(P):
    kv = inputs.paged_kv(1160 + P, [1000, 3 * P + 2], Hkv=8, page_size=P, fill_unused="normal")
    check_attention(kv, inputs.query(1160 + P, 2, 16), 0)


def test_int8_attention_empty_context_and_bad_page_flags():
    kv = inputs.paged_kv(1170, [40, 40], Hkv=8, page_size=16, fill_unused="normal")
    kv.context_lens[0] = 0
    kv.block_table[1, 2] = kv.num_pages + 9
    k8, v8, ks, vs = int8_cache(kv)
    of, _ = run_attention(kv, inputs.query(1170, 2, 16), k8, v8, ks, vs)
    assert pg.device_error_flags() & binding.DEVERR_BAD_PAGE
    assert np.all(of[0] == 0) and np.isfinite(of).all()


def test_int8_prologue_matches_the_oracle():
    ctx = [40, 17, 64, 1]
    B = len(ctx)
    kv = inputs.paged_kv(1180, ctx, Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(1180, B, 16, 8)
    k8, v8, ks, vs = (np.nan_to_num(a) for a in int8_cache(kv))
    dev = "cuda"
    dk8, dv8, dks, dvs = dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs)
    q_out = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append_int8(to_device_bf16(tok.q, dev), to_device_bf16(tok.k, dev), to_device_bf16(tok.v, dev),
                                to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev),
                                to_device_i32(kv.context_lens, dev), to_device_i32(kv.block_table, dev), dk8, dv8,
                                dks, dvs, q_out, THETA)
    torch.cuda.synchronize()
    q_ref, k8r, v8r, ksr, vsr = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, THETA)
    assert_bf16_close(bf16_bits(q_out), q_ref, "q_out")
    gk8, gv8, gks, gvs = dk8.cpu().numpy(), dv8.cpu().numpy(), dks.cpu().numpy(), dvs.cpu().numpy()
    # V is quantized from the same bf16 row: codes and scales bit for bit
    assert np.array_equal(gv8, v8r) and np.array_equal(gvs, vsr)
    # K from the rotated row, whose bf16 rounding may differ by 1 ulp: only the
    # appended rows change, their codes within 1 step and scales within 2^-7
    changed = np.any(gk8 != k8, axis=-1) | np.any(k8r != k8, axis=-1) | (gks != ks) | (ksr != ks)
    assert np.array_equal(gk8[~changed], k8[~changed]) and np.array_equal(gks[~changed], ks[~changed])
    assert np.abs(gk8.astype(np.int32) - k8r.astype(np.int32)).max() <= 1
    assert np.all(np.abs(gks - ksr) <= np.abs(ksr) * 2.0 ** -7)
    assert pg.device_error_flags() == 0


def test_int8_prologue_then_attention_chain():
    ctx = [300, 17, 2049]
    B = len(ctx)
    kv = inputs.paged_kv(1190, ctx, Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(1190, B, 16, 8)
    k8, v8, ks, vs = (np.nan_to_num(a) for a in int8_cache(kv))
    dev = "cuda"
    dk8, dv8, dks, dvs = dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs)
    bt, cl = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
    q_out = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.qk_norm_rope_append_int8(to_device_bf16(tok.q, dev), to_device_bf16(tok.k, dev), to_device_bf16(tok.v, dev),
                                to_device_bf16(tok.gamma_q, dev), to_device_bf16(tok.gamma_k, dev), cl, bt, dk8, dv8,
                                dks, dvs, q_out, THETA)
    n = pg.decode_attn_int8_workspace_size(B, 16, 8, 128, 16, kv.max_pages, 0)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    of = torch.empty((B, 16, 128), dtype=torch.float32, device=dev)
    ob = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=dev)
    pg.decode_attn_paged_int8(q_out, dk8, dv8, dks, dvs, bt, cl, SCALE, out_f32=of, out_bf16=ob, workspace=ws)
    torch.cuda.synchronize()
    q_ref, k8r, v8r, ksr, vsr = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, THETA)
    ref = oracle.decode_attention_int8(q_ref, k8r, v8r, ksr, vsr, kv.block_table, kv.context_lens, SCALE)
    assert np.abs(of.cpu().numpy() - ref).max() <= ATOL_F32
    own = oracle.decode_attention_int8(bf16_bits(q_out), dk8.cpu().numpy(), dv8.cpu().numpy(), dks.cpu().numpy(),
                                       dvs.cpu().numpy(), kv.block_table, kv.context_lens, SCALE)
    assert_bf16_close(bf16_bits(ob), oracle.round_bf16(own), "out_bf16")
    assert pg.device_error_flags() == 0


def test_int8_quality_gate_against_bf16_attention():
    """INT8 rows (symmetric per row, 8 bits) against the bf16 cache they came
    from, on N(0,1) keys and values: the attention output stays within 2 %
    RMS relative error and 0.05 absolute (a bf16 row has 8 significant bits,
    an INT8 row about 7 relative to its largest element)."""
    ctx = [4096, 333, 8000]
    kv = inputs.paged_kv(1200, ctx, Hkv=8, page_size=16, fill_unused="normal")
    q = inputs.query(1200, len(ctx), 16)
    k8, v8, ks, vs = int8_cache(kv)
    of, _ = run_attention(kv, q, k8, v8, ks, vs)
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
    rms = math.sqrt(float(((of - ref) ** 2).mean() / (ref ** 2).mean()))
    print(f"INT8 vs bf16 attention: RMS relative {rms:.4f}, max abs {np.abs(of - ref).max():.4f}")
    assert rms <= 0.02
    assert np.abs(of - ref).max() <= 0.05


def _fused_vs_two_launch(seed, ctx, Hq, num_partitions, page_size=16):
    """Runs decode_step_paged_int8 and the prologue + attention pair on copies
    of the same INT8 cache; returns both results and the oracle inputs."""
    B, Hkv = len(ctx), 8
    kv = inputs.paged_kv(seed, ctx, Hkv=Hkv, page_size=page_size, fill_unused="normal")
    tok = inputs.new_token(seed, B, Hq, Hkv)
    k8, v8, ks, vs = (np.nan_to_num(a) for a in int8_cache(kv))
    dev = "cuda"
    bt, cl = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
    raw = [to_device_bf16(a, dev) for a in (tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k)]
    n = pg.decode_attn_int8_workspace_size(B, Hq, Hkv, 128, page_size, kv.max_pages, num_partitions)
    res = {}
    for mode in ("fused", "two"):
        cache = [dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs)]
        ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
        q_out = torch.full((B, Hq, 128), 0x7FC0, dtype=torch.int16, device=dev).view(torch.bfloat16)
        of = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        ob = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16, device=dev)
        if mode == "fused":
            pg.decode_step_paged_int8(*raw, cl, bt, *cache, SCALE, THETA, q_out=q_out, out_f32=of, out_bf16=ob,
                                      workspace=ws, num_partitions=num_partitions)
        else:
            pg.qk_norm_rope_append_int8(*raw, cl, bt, *cache, q_out, THETA)
            pg.decode_attn_paged_int8(q_out, *cache, bt, cl, SCALE, out_f32=of, out_bf16=ob, workspace=ws,
                                      num_partitions=num_partitions)
        torch.cuda.synchronize()
        res[mode] = [t.cpu().numpy() for t in cache] + [bf16_bits(q_out), of.cpu().numpy(), bf16_bits(ob)]
    return res, kv, tok, (k8, v8, ks, vs)


@pytest.mark.parametrize("ctx,Hq,num_partitions", [
    ([1, 16, 17, 300], 16, 0),
    ([2049, 40, 8000], 16, 0),
    ([2049, 40, 8000], 16, 70),
    ([700, 1], 64, 5),
    ([2049, 40, 3000], 64, 24),
    ([12000, 11000, 9000, 12000, 5000, 12000, 7], 16, 3),
    ([512, 513], 8, 1),
])
def test_int8_fused_step_equals_two_launches(ctx, Hq, num_partitions):
    """decode_step_paged_int8 writes the same codes and scales, the same
    rotated query and the same outputs (bit for bit) as the quantizing
    prologue followed by the INT8 attention (one and several CTAs per SM:
    70 partitions of g = 2 run four per SM, 24 of g = 8 two per SM, and so
    do 3 partitions of 4000 positions over 7 sequences)."""
    res, *_ = _fused_vs_two_launch(1300 + sum(ctx) % 97 + Hq, ctx, Hq, num_partitions)
    for name, a, b in zip(("k8", "v8", "k_scale", "v_scale", "q_out", "out_f32", "out_bf16"), res["fused"], res["two"]):
        assert np.array_equal(a, b, equal_nan=False), name
    assert pg.device_error_flags() == 0


@pytest.mark.parametrize("num_partitions", [0, 3])
def test_int8_fused_step_matches_the_oracle(num_partitions):
    ctx = [300, 17, 2049, 1]
    res, kv, tok, (k8, v8, ks, vs) = _fused_vs_two_launch(1320 + num_partitions, ctx, 16, num_partitions)
    q_ref, k8r, v8r, ksr, vsr = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, THETA)
    ref = oracle.decode_attention_int8(q_ref, k8r, v8r, ksr, vsr, kv.block_table, kv.context_lens, SCALE)
    gk8, gv8, gks, gvs, gq, of, ob = res["fused"]
    assert np.abs(of - ref).max() <= ATOL_F32
    assert_bf16_close(gq, q_ref, "q_out")
    assert np.array_equal(gv8, v8r) and np.array_equal(gvs, vsr)
    own = oracle.decode_attention_int8(gq, gk8, gv8, gks, gvs, kv.block_table, kv.context_lens, SCALE)
    assert_bf16_close(ob, oracle.round_bf16(own), "out_bf16")
    assert pg.device_error_flags() == 0


@pytest.mark.parametrize("Hq,num_partitions", [(8, 64), (24, 28), (24, 32), (48, 40)])
def test_int8_several_ctas_per_sm(Hq, num_partitions):
    """Several waves of short partitions (8 sequences x 8 KV heads x 26-64
    partitions of 32-80 positions) run several CTAs per SM: four of 4 warps
    (48 KiB of stages each) for g = 1 and 3, two of 8 warps for g = 6. The
    last CTA merges g = 1 at 64 partitions and g = 3 at 26 (28 asked); g = 3
    at 32 and g = 6 at 32 (40 asked) do not fit and merge in merge_kernel.
    Attention against the oracle's INT8 attention, the fused step against the
    oracle's chain and bit for bit against the two launches."""
    ctx = [2048, 1, 2, 1500, 2047, 700, 2048, 33]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    max_pages = 128
    np_used = pg.decode_attn_partition_count(len(ctx), 8, 16, max_pages, num_partitions)
    assert len(ctx) * 8 * np_used > sms and -(-max_pages // np_used) * 16 <= 2048
    kv = inputs.paged_kv(1400 + Hq, ctx, Hkv=8, page_size=16, fill_unused="normal")
    assert kv.max_pages == max_pages
    check_attention(kv, inputs.query(1400 + Hq, len(ctx), Hq), num_partitions)
    res, kv, tok, (k8, v8, ks, vs) = _fused_vs_two_launch(1410 + Hq, ctx, Hq, num_partitions)
    for name, a, b in zip(("k8", "v8", "k_scale", "v_scale", "q_out", "out_f32", "out_bf16"), res["fused"], res["two"]):
        assert np.array_equal(a, b, equal_nan=False), name
    q_ref, k8r, v8r, ksr, vsr = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, THETA)
    ref = oracle.decode_attention_int8(q_ref, k8r, v8r, ksr, vsr, kv.block_table, kv.context_lens, SCALE)
    gk8, gv8, gks, gvs, gq, of, ob = res["fused"]
    assert np.abs(of - ref).max() <= ATOL_F32
    own = oracle.decode_attention_int8(gq, gk8, gv8, gks, gvs, kv.block_table, kv.context_lens, SCALE)
    assert_bf16_close(ob, oracle.round_bf16(own), "out_bf16")
    assert pg.device_error_flags() == 0


def test_int8_fused_step_flags_empty_context_and_bad_page():
    """T = 0 cannot hold the new token: zeros and the context flag. A new
    position whose page lies outside the pool is not written: page flag."""
    kv = inputs.paged_kv(1330, [40, 40], Hkv=8, page_size=16, fill_unused="normal")
    kv.context_lens[0] = 0
    kv.block_table[1, 2] = kv.num_pages + 9  # the page of position 39
    tok = inputs.new_token(1330, 2, 16, 8)
    k8, v8, ks, vs = (np.nan_to_num(a) for a in int8_cache(kv))
    dev = "cuda"
    cache = [dev_i8(k8), dev_i8(v8), dev_f32(ks), dev_f32(vs)]
    n = pg.decode_attn_int8_workspace_size(2, 16, 8, 128, 16, kv.max_pages, 0)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    of = torch.full((2, 16, 128), float("nan"), dtype=torch.float32, device=dev)
    raw = [to_device_bf16(a, dev) for a in (tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k)]
    pg.decode_step_paged_int8(*raw, to_device_i32(kv.context_lens, dev), to_device_i32(kv.block_table, dev), *cache,
                              SCALE, THETA, out_f32=of, workspace=ws)
    flags = pg.device_error_flags()
    assert flags & binding.DEVERR_BAD_CONTEXT and flags & binding.DEVERR_BAD_PAGE
    out = of.cpu().numpy()
    assert np.all(out[0] == 0) and np.isfinite(out).all()
    assert np.array_equal(cache[0].cpu().numpy(), k8) and np.array_equal(cache[2].cpu().numpy(), ks)


def test_int8_fused_step_full_size_t8192():
    """One layer of the Qwen3-0.6B-shaped step (B = 1, Hq = 16, Hkv = 8,
    T = 8192, P = 16) over an INT8 cache, in the launch configuration the
    benchmark times (automatic partition count), against the oracle's INT8
    prologue and attention on every output."""
    res, kv, tok, (k8, v8, ks, vs) = _fused_vs_two_launch(1340, [8192], 16, 0)
    q_ref, k8r, v8r, ksr, vsr = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, THETA)
    ref = oracle.decode_attention_int8(q_ref, k8r, v8r, ksr, vsr, kv.block_table, kv.context_lens, SCALE)
    gk8, gv8, gks, gvs, gq, of, ob = res["fused"]
    assert np.abs(of - ref).max() <= ATOL_F32
    own = oracle.decode_attention_int8(gq, gk8, gv8, gks, gvs, kv.block_table, kv.context_lens, SCALE)
    assert_bf16_close(ob, oracle.round_bf16(own), "out_bf16")
    for name, a, b in zip(("k8", "v8", "k_scale", "v_scale", "q_out", "out_f32", "out_bf16"), res["fused"], res["two"]):
        assert np.array_equal(a, b), name
    assert pg.device_error_flags() == 0


def _carved(first, second):
    """Two device tensors carved from one allocation, `first` at the lower
    address (so the order of the code caches and of the scale arrays in
    memory is fixed)."""
    a = np.ascontiguousarray(first)
    b = np.ascontiguousarray(second)
    buf = torch.from_numpy(np.concatenate([a.reshape(-1).view(np.uint8), b.reshape(-1).view(np.uint8)])).cuda()
    n = a.nbytes
    return (buf[:n].view(torch.int8 if a.dtype == np.int8 else torch.float32).view(a.shape),
            buf[n:].view(torch.int8 if b.dtype == np.int8 else torch.float32).view(b.shape))


@pytest.mark.parametrize("v_first", [False, True])
def test_int8_attention_with_either_order_of_the_caches_in_memory(v_first):
    """V above K in memory lets one copy fetch a chunk's K and V codes (and
    one its scales); V below K takes the separate copies. Both give the
    same bits, and the oracle's attention."""
    kv = inputs.paged_kv(1190, [3000, 700], Hkv=8, page_size=16, fill_unused="normal")
    q = inputs.query(1190, 2, 16)
    k8, v8, ks, vs = int8_cache(kv)
    B, Hq = 2, 16
    if v_first:
        v8d, k8d = _carved(v8, k8)
        vsd, ksd = _carved(vs, ks)
    else:
        k8d, v8d = _carved(k8, v8)
        ksd, vsd = _carved(ks, vs)
    outs = []
    for npr in (0, 5):
        n = pg.decode_attn_int8_workspace_size(B, Hq, 8, 128, kv.page_size, kv.max_pages, npr)
        ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
        of = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        pg.decode_attn_paged_int8(to_device_bf16(q, "cuda"), k8d, v8d, ksd, vsd, to_device_i32(kv.block_table, "cuda"),
                                  to_device_i32(kv.context_lens, "cuda"), SCALE, out_f32=of, workspace=ws,
                                  num_partitions=npr)
        torch.cuda.synchronize()
        outs.append(of.cpu().numpy())
    ref = oracle.decode_attention_int8(q, k8, v8, ks, vs, kv.block_table, kv.context_lens, SCALE)
    for o in outs:
        assert np.abs(o - ref).max() <= ATOL_F32
    # the same bits as the default allocation (each cache its own tensor)
    for o, npr in zip(outs, (0, 5)):
        of, _ = run_attention(kv, q, k8, v8, ks, vs, npr)
        assert np.array_equal(o, of)
    assert pg.device_error_flags() == 0
