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
