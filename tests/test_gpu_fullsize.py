"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times. Where the oracle would be too slow for every output, a
seeded sample of sequences is checked one by one and properties that hold at
any size are checked for the rest."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import inputs
from parity_util import assert_bf16_close
from paged_gqa_decode_head_gb300.runner import DecodeStep, bf16_bits, to_device_bf16, to_device_i32

pytestmark = pytest.mark.gpu

ATOL_F32 = 2e-3
SCALE = 1.0 / math.sqrt(128)


@pytest.mark.parametrize("fused", [True, False])
def test_qwen3_28_layer_step_t8192_graph(fused):
    """The benchmark's step (fused: one decode_step_paged launch per layer;
    otherwise qk_norm_rope_append + decode_attn_paged) replayed as one graph."""
    w = inputs.WORKLOADS["qwen3_0p6b_t8k"]
    layers = inputs.qwen3_layers()
    step = DecodeStep(layers, Hq=w["Hq"], Hkv=w["Hkv"], rope_theta=w["theta"])
    step.capture(fused=fused)
    step.replay()
    torch.cuda.synchronize()
    assert pg.device_error_flags() == 0
    worst = 0.0
    for (kv, tok), st in zip(layers, step.layers):
        q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                           kv.context_lens, kv.block_table, kv.k_cache, kv.v_cache,
                                                           kv.page_size, w["theta"])
        assert_bf16_close(bf16_bits(st.q_out), q_ref)
        ref = oracle.decode_attention(q_ref, kc_ref, vc_ref, kv.block_table, kv.context_lens, SCALE)
        err = np.abs(st.out_f32.cpu().numpy().astype(np.float64) - ref).max()
        worst = max(worst, err)
        assert err <= ATOL_F32
        # the bf16 output is the nearest-even cast of the fp32 output
        assert np.array_equal(bf16_bits(st.out_bf16), oracle.round_bf16(st.out_f32.cpu().numpy()))
    print(f"28 layers: worst |out - oracle| = {worst:.2e}")
    # replaying the step reproduces every output bit for bit (the appends
    # rewrite the same rows; the fold grouping never depends on timing)
    first = step.outputs.clone()
    for _ in range(3):
        step.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.outputs, first)


def test_ragged_b64_full_size_sampled():
    w = inputs.WORKLOADS["ragged_b64"]
    kv, q = inputs.ragged_b64()
    dev = "cuda"
    B = w["B"]
    qd = to_device_bf16(q, dev)
    kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
    bt, ctx = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
    ws = torch.zeros(max(16, pg.decode_attn_workspace_size(B, w["Hq"], w["Hkv"], 128, 16, kv.max_pages, 0)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, w["Hq"], 128), dtype=torch.float32, device=dev)
    pg.decode_attn_paged(qd, kc, vc, bt, ctx, SCALE, out_f32=out, workspace=ws)
    torch.cuda.synchronize()
    assert pg.device_error_flags() == 0
    o = out.cpu().numpy()
    assert np.isfinite(o).all()
    # a convex combination of unit-normal V rows stays well inside their range
    assert np.abs(o).max() < 6.0
    order = np.argsort(kv.context_lens)
    sample = sorted({int(order[0]), int(order[-1]), *np.random.default_rng(5).choice(B, 4, replace=False).tolist()})
    for b in sample:
        ref = oracle.decode_attention(q[b:b + 1], kv.k_cache, kv.v_cache, kv.block_table[b:b + 1],
                                      kv.context_lens[b:b + 1], SCALE)
        assert np.abs(o[b:b + 1] - ref).max() <= ATOL_F32, b


def test_long_split_kv_t131072_np256():
    w = inputs.WORKLOADS["long_split_kv_t128k"]
    kv, q = inputs.long_split_kv()
    dev = "cuda"
    np_req = w["T"] // w["partition"]
    assert pg.decode_attn_partition_count(1, w["Hkv"], 16, kv.max_pages, np_req) == 256
    ws = torch.zeros(pg.decode_attn_workspace_size(1, w["Hq"], w["Hkv"], 128, 16, kv.max_pages, np_req),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((1, w["Hq"], 128), dtype=torch.float32, device=dev)
    outb = torch.empty((1, w["Hq"], 128), dtype=torch.bfloat16, device=dev)
    pg.decode_attn_paged(to_device_bf16(q, dev), to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev),
                         to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev), SCALE,
                         out_f32=out, out_bf16=outb, workspace=ws, num_partitions=np_req)
    torch.cuda.synchronize()
    assert pg.device_error_flags() == 0
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, SCALE)
    assert np.abs(out.cpu().numpy() - ref).max() <= ATOL_F32
    assert_bf16_close(bf16_bits(outb), oracle.round_bf16(ref))


@pytest.mark.parametrize("tiles_per_copy", [1, 8])
def test_host_tiled_t65536(tiles_per_copy):
    """The host-tiled workload: 128 tiles of 512 positions, copied one tile
    per copy (the pages' pipeline) or eight per copy, as the benchmark runs
    them."""
    w = inputs.WORKLOADS["host_tiled_t64k"]
    q, k, v = inputs.host_tiled_kv()
    dev = "cuda"
    B, Hq, Hkv, tile = w["B"], w["Hq"], w["Hkv"], w["tile"]
    hk = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
    span = tile * tiles_per_copy
    slots_k = [torch.empty((B, span, Hkv, 128), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    slots_v = [torch.empty((B, span, Hkv, 128), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    events = [torch.cuda.Event() for _ in range(4)]
    m = torch.empty((B, Hq), device=dev)
    l = torch.empty((B, Hq), device=dev)
    acc = torch.empty((B, Hq, 128), device=dev)
    out = torch.empty((B, Hq, 128), device=dev)
    pg.attn_host_tiled_run(to_device_bf16(q, dev), hk, hv, SCALE, slots_k, slots_v, events, m, l, acc,
                           out_f32=out, tile_len=tile, tiles_per_copy=tiles_per_copy, copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    ref = oracle.attention_contiguous(q, k, v, SCALE)
    assert np.abs(out.cpu().numpy() - ref).max() <= ATOL_F32
