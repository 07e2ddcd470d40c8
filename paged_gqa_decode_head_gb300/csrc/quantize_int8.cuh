// quantize_int8.cuh -- symmetric per-row INT8 quantization of one head row
// held by a warp (lane l holds dims l, l+32, l+64, l+96).
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime" s0.1: INT8
// values carry one FP32 scale and are read back as code x scale. A KV row is
// one (position, KV head) vector of 128 values: s = amax / 127 and code =
// round_half_even(x / s), both in binary32 with correctly rounded division;
// an all-zero row has s = 0 and codes 0. Shared by the prologue and the fused
// INT8 decode step so both write the same bytes.
#pragma once

#include "common.cuh"

namespace pgqa {

// Warp-collective: returns s and this lane's four codes (dims lane + 32 i).
__device__ __forceinline__ float quantize_head_int8(const float (&x)[4], int (&code)[4])
{
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        code[i] = amax > 0.0f ? max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], s)))) : 0;
    return s;
}

// Quantizes the warp's row and stores its 128 codes and its scale.
__device__ __forceinline__ void store_row_int8(const float (&x)[4], int8_t *codes, float *scale)
{
    const int lane = threadIdx.x & 31;
    int c[4];
    const float s = quantize_head_int8(x, c);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        codes[lane + 32 * i] = static_cast<int8_t>(c[i]);
    if (lane == 0)
        *scale = s;
}

// The bf16 rounding of a rotated K row, which is what the INT8 cache
// quantizes (the bf16 cache would hold exactly these values).
__device__ __forceinline__ void round_head_bf16(float (&x)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
        x[i] = bf16_bits_to_f32(f32_to_bf16_bits(x[i]));
}

} // namespace pgqa
