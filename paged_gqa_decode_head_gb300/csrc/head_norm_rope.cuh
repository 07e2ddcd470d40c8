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

#include "common.cuh"

namespace pgqa {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h)
{
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Rotate the pair (a, b) whose frequency is inv_freq at position pos.
__device__ __forceinline__ void rope_pair(float &a, float &b, int pos, double inv_freq)
{
    // 2*pi as an unevaluated sum hi + lo of two doubles.
    constexpr double kTwoPiHi = 6.283185307179586232;
    constexpr double kTwoPiLo = 2.4492935982947064e-16;
    constexpr double kInvTwoPi = 0.15915494309189535;
    const double phi = static_cast<double>(pos) * inv_freq;
    const double n = rint(phi * kInvTwoPi);
    double r = fma(-n, kTwoPiHi, phi);
    r = fma(-n, kTwoPiLo, r);
    float sn, cs;
    sincosf(static_cast<float>(r), &sn, &cs);
    const float ra = a * cs - b * sn;
    const float rb = b * cs + a * sn;
    a = ra;
    b = rb;
}

// x[i] (dim lane + 32 i) of RoPE_pos(RMSNorm(src) * gamma); whole warp.
// inv_freq[i] = theta^(-2i/128) for i < 64.
__device__ __forceinline__ void norm_rope_head(const uint16_t *src, const uint16_t *gamma, float eps,
                                               int pos, const double *inv_freq, float (&x)[4])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        x[i] = bf16_bits_to_f32(src[lane + 32 * i]);
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    const float inv_rms = rsqrtf(ss * (1.0f / kHeadDim) + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        x[i] = x[i] * inv_rms * bf16_bits_to_f32(gamma[lane + 32 * i]);
    // pairs (lane, lane + 64) and (lane + 32, lane + 96)
    rope_pair(x[0], x[2], pos, inv_freq[lane]);
    rope_pair(x[1], x[3], pos, inv_freq[lane + 32]);
}

} // namespace pgqa
