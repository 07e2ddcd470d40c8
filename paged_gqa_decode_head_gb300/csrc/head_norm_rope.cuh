// head_norm_rope.cuh -- one warp normalises and rotates one 128-dim head.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime":
//   s2.3 per-head RMSNorm with learned gains (s2.1: eps);
//   s2.4 RoPE rotates the pair (x_i, x_{i+D/2}) by pos * theta^(-2i/D);
//   s7.1 one warp per head: lane l holds dims l, l+32, l+64, l+96, so both
//        RoPE pairs (l, l+64) and (l+32, l+96) are in-lane and the norm is a
//        5-step shuffle reduction.
// The phase pos * omega_i is formed in fp64 (omega_i given in fp64) and
// reduced modulo 2*pi before the fp32 sincosf, so the angle stays accurate
// to ~1e-7 rad even at pos ~ 1e5 where an fp32 product would be off by ~1e-2.
#pragma once

#include <cmath>

#include "common.cuh"

namespace pgqa {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h)
{
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// cos and sin of the RoPE angle pos * inv_freq, the angle reduced modulo
// 2*pi in fp64 first.
__device__ __forceinline__ void rope_angle(int pos, double inv_freq, float &cs, float &sn)
{
    // 2*pi as an unevaluated sum hi + lo of two doubles.
    constexpr double kTwoPiHi = 6.283185307179586232;
    constexpr double kTwoPiLo = 2.4492935982947064e-16;
    constexpr double kInvTwoPi = 0.15915494309189535;
    const double phi = static_cast<double>(pos) * inv_freq;
    const double n = rint(phi * kInvTwoPi);
    double r = fma(-n, kTwoPiHi, phi);
    r = fma(-n, kTwoPiLo, r);
    sincosf(static_cast<float>(r), &sn, &cs);
}

// The RoPE frequencies omega_i = theta^(-2i/128) as r^i, r = theta^(-2/128),
// from the six powers r^(2^k) (k = 0..5): lane l forms omega_l and
// omega_(l+32) with at most six fp64 products (relative error ~1e-15), and
// every lane reads the same six values, which a per-lane table index into
// kernel parameters would serialise.
struct RopeFreqs {
    double r_pow2[6]; // r^(2^k)
};

inline RopeFreqs make_rope_freqs(double theta)
{
    RopeFreqs f;
    for (int k = 0; k < 6; ++k)
        f.r_pow2[k] = std::pow(theta, -2.0 * (1 << k) / kHeadDim);
    return f;
}

// The rotation of this lane's two pairs (lane, lane + 64) and
// (lane + 32, lane + 96) at position pos.
struct HeadRope {
    float cs[2], sn[2];
    __device__ __forceinline__ void init(int pos, const RopeFreqs &f)
    {
        const int lane = threadIdx.x & 31;
        double w = 1.0;
#pragma unroll
        for (int k = 0; k < 5; ++k)
            if ((lane >> k) & 1)
                w *= f.r_pow2[k];
        rope_angle(pos, w, cs[0], sn[0]);
        rope_angle(pos, w * f.r_pow2[5], cs[1], sn[1]);
    }
};

// This lane's four elements (dims lane + 32 i) of a bf16 head vector.
__device__ __forceinline__ void load_head(const uint16_t *src, float (&x)[4])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        x[i] = bf16_bits_to_f32(src[lane + 32 * i]);
}

// x <- RoPE(RMSNorm(x) * gain) for the head held by the warp (x[i] is dim
// lane + 32 i). Every product and sum is rounded explicitly (no contraction
// left to the compiler), so every kernel that uses this gets the same bits.
__device__ __forceinline__ void norm_rope_apply(float (&x)[4], const float (&gain)[4], float eps,
                                                const HeadRope &rope)
{
    float ss = __fmul_rn(x[0], x[0]);
    ss = __fmaf_rn(x[1], x[1], ss);
    ss = __fmaf_rn(x[2], x[2], ss);
    ss = __fmaf_rn(x[3], x[3], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
    const float inv_rms = rsqrtf(__fadd_rn(__fmul_rn(ss, 1.0f / kHeadDim), eps));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        x[i] = __fmul_rn(__fmul_rn(x[i], inv_rms), gain[i]);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float a = x[j], b = x[j + 2];
        x[j] = __fmaf_rn(a, rope.cs[j], -__fmul_rn(b, rope.sn[j]));
        x[j + 2] = __fmaf_rn(b, rope.cs[j], __fmul_rn(a, rope.sn[j]));
    }
}

// x[i] (dim lane + 32 i) of RoPE_pos(RMSNorm(src) * gamma); whole warp.
__device__ __forceinline__ void norm_rope_head(const uint16_t *src, const uint16_t *gamma, float eps,
                                               int pos, const RopeFreqs &freqs, float (&x)[4])
{
    HeadRope rope;
    rope.init(pos, freqs);
    float gain[4];
    load_head(gamma, gain);
    load_head(src, x);
    norm_rope_apply(x, gain, eps, rope);
}

} // namespace pgqa
