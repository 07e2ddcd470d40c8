"""GPU parity of attn_host_direct, the zero-copy variant of the host-tiled
attention: the history stays in pinned host memory and the kernel reads it
directly; compared with the oracle's full-softmax attention over the same
contiguous history."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_head_gb300 as pg
from paged_gqa_decode_head_gb300 import binding, inputs
from paged_gqa_decode_head_gb300.runner import bf16_bits, to_device_bf16
from parity_util import assert_bf16_close

pytestmark = pytest.mark.gpu

ATOL_F32 = 2e-3
SCALE = 1.0 / math.sqrt(128)


def _pinned(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


def run_direct(q, k, v, num_partitions=0):
    B, Hq, _ = q.shape
    _, T, Hkv, _ = k.shape
    hk, hv = _pinned(k), _pinned(v)
    n = pg.attn_host_direct_workspace_size(B, Hq, Hkv, T, num_partitions)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    of = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ob = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pg.attn_host_direct(to_device_bf16(q, "cuda"), hk, hv, SCALE, out_f32=of, out_bf16=ob, workspace=ws,
                        num_partitions=num_partitions)
    torch.cuda.synchronize()
    return of.cpu().numpy(), bf16_bits(ob)


def check(seed, B, T, Hq, Hkv, num_partitions=0):
    q = inputs.query(seed, B, Hq, 128)
    k, v = inputs.contiguous_kv(seed, B, T, Hkv)
    of, ob = run_direct(q, k, v, num_partitions)
    ref = oracle.attention_contiguous(q, k, v, SCALE)
    assert np.isfinite(of).all()
    assert np.abs(of - ref).max() <= ATOL_F32
    assert_bf16_close(ob, oracle.round_bf16(ref), "out_bf16")


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 511, 512, 513, 1000])
def test_host_direct_small_contexts(T):
    check(500 + T, 2, T, 16, 8)


@pytest.mark.parametrize("num_partitions", [1, 2, 7, 100])
def test_host_direct_partition_counts(num_partitions):
    check(520 + num_partitions, 1, 3000, 16, 8, num_partitions)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (24, 8), (32, 8), (64, 8), (4, 1)])
def test_host_direct_group_sizes(Hq, Hkv):
    check(540 + Hq, 3, 700, Hq, Hkv, 5)


def test_host_direct_empty_history_gives_zeros():
    q = inputs.query(560, 2, 16, 128)
    k = np.zeros((2, 0, 8, 128), dtype=np.uint16)
    of, ob = run_direct(q, k, k.copy())
    assert np.all(of == 0) and np.all(ob == 0)


def test_host_direct_full_size_t65536():
    """The host-tiled workload (T = 65536, 256 MiB in pinned host memory),
    read in place instead of tile by tile."""
    w = inputs.WORKLOADS["host_tiled_t64k"]
    q, k, v = inputs.host_tiled_kv()
    of, ob = run_direct(q, k, v)
    ref = oracle.attention_contiguous(q, k, v, SCALE)
    assert np.abs(of - ref).max() <= ATOL_F32
    assert_bf16_close(ob, oracle.round_bf16(ref), "out_bf16")
    assert pg.attn_host_direct_partition_count(w["B"], w["Hkv"], w["T"]) >= 2


def test_host_direct_refuses_unmapped_history():
    """Pageable host memory is refused before any launch (or, where the
    platform maps it anyway, read correctly)."""
    B, T, Hq, Hkv = 1, 64, 16, 8
    q = inputs.query(570, B, Hq, 128)
    k, v = inputs.contiguous_kv(570, B, T, Hkv)
    kp = np.ascontiguousarray(k)
    vp = np.ascontiguousarray(v)
    qd = to_device_bf16(q, "cuda")
    of = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    lib = binding.load_library()
    rc = lib.attn_host_direct(qd.data_ptr(), kp.ctypes.data_as(ctypes.c_void_p), vp.ctypes.data_as(ctypes.c_void_p),
                              T, B, Hq, Hkv, 128, ctypes.c_float(SCALE), 1, of.data_ptr(), None, None, 0, None)
    torch.cuda.synchronize()
    if rc == 0:
        ref = oracle.attention_contiguous(q, k, v, SCALE)
        assert np.abs(of.cpu().numpy() - ref).max() <= ATOL_F32
    else:
        assert rc == -1
        assert b"mapped" in lib.pgqa_last_error()
