"""Comparison helpers shared by the GPU parity tests.

bf16 bar: the GPU's bf16 result and the oracle's nearest-even rounding of its
fp64 result may differ by at most 1 bf16 ulp. Below 2^-10 the absolute error
of the computation, not the cast, sets the achievable accuracy: the attention
weights p enter the P.V product as a bf16 hi + lo pair (about 16 significant
bits, relative error up to 2^-17 per weight), which leaves an absolute error
of order 2^-17 times the magnitude of V on every output; the fp32
accumulation adds about 1e-7. So there the ulp is counted as that of 2^-10
(2^-17 absolute).
"""
import numpy as np
import torch

import paged_gqa_decode_head_gb300 as pg

BF16_ULP_FLOOR = 2.0 ** -17  # one bf16 ulp at 2^-10


def ordered(bits):
    """bf16 bit patterns -> integers monotone in the value (+0 and -0 coincide)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_diff(a, b):
    return np.abs(ordered(a) - ordered(b))


def widen(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_within_one_ulp(gpu_bits, ref_bits):
    """True where the two bf16 values differ by <= 1 ulp (ulp floored at 2^-10)."""
    close = ulp_diff(gpu_bits, ref_bits) <= 1
    tiny = np.abs(widen(gpu_bits) - widen(ref_bits)) <= BF16_ULP_FLOOR
    return close | tiny


def assert_bf16_close(gpu_bits, ref_bits, what="bf16"):
    ok = bf16_within_one_ulp(gpu_bits, ref_bits)
    if not ok.all():
        idx = np.argwhere(~ok)[0]
        g = widen(gpu_bits)[tuple(idx)]
        r = widen(ref_bits)[tuple(idx)]
        raise AssertionError(f"{what}: {int((~ok).sum())} values beyond 1 ulp, first at {tuple(idx)}: "
                             f"gpu {g!r} vs oracle {r!r}")


def walked(B, Hq, Hkv, P, max_pages, num_partitions):
    """The library's rule for walking partitions (decode_walk_kernel): attention
    alone over a grid of the two-CTA shape (one new token, g <= 6, more CTAs
    than SMs, partitions of at most 2048 positions) with g <= 4, whose states
    the merge kernel merges (over 64 partitions, or more accumulators than its
    96 KiB of stages hold beside 5184 bytes of scratch), and few enough
    (sequence, KV head) pairs that runs of partitions fill at least 7/8 of the
    CTA slots (two per SM)."""
    np_used = pg.decode_attn_partition_count(B, Hkv, P, max_pages, num_partitions)
    ppp = -(-max_pages // np_used)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = Hq // Hkv
    pair = G <= 6 and np_used > 1 and ppp * P <= 2048 and B * Hkv * np_used > sms
    merge_kernel = np_used > 64 or G * np_used * 128 * 4 + 5184 > 6 * 2 * 8192
    heads = B * Hkv
    slots = 2 * sms
    per_head = slots // heads
    return (pair and G <= 4 and merge_kernel and heads <= slots and per_head * heads * 8 >= slots * 7
            and -(-np_used // max(1, per_head)) >= 2)
