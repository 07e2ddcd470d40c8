// prologue.cu -- fused per-head Q/K RMSNorm + half-rotation RoPE + paged K/V
// append for the decode step.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime":
//   s2.3 per-head RMSNorm of Q and K with learned gains (s2.1: eps), V is
//        not normalised;
//   s2.4 RoPE rotates the pair (x_i, x_{i+D/2}) by pos * theta^(-2i/D);
//   s7.1 one warp per head: lane l holds dims l, l+32, l+64, l+96, so both
//        RoPE pairs (l, l+64) and (l+32, l+96) are in-lane and the norm is
//        a 5-step shuffle reduction;
//   s7.2 the rotated K goes straight to its physical page
//        block_table[b][pos / P] at offset pos % P.
//
// The norm and rotation of one head are in head_norm_rope.cuh (shared with
// the fused decode step).
#include "common.cuh"
#include "head_norm_rope.cuh"
#include "launch.h"
#include "quantize_int8.cuh"

namespace pgqa {
namespace {

__device__ unsigned g_flags_prologue;

constexpr int kWarpsPerBlock = 4;

struct PrologueParams {
    const uint16_t *q, *k, *v, *gamma_q, *gamma_k;
    const int32_t *context_lens, *block_table;
    uint16_t *k_cache, *v_cache, *q_out;
    // INT8 cache (kInt8): codes [num_pages][Hkv][P][D] and one FP32 scale per row
    int8_t *k_cache8, *v_cache8;
    float *k_scale, *v_scale;
    int B, M, Hq, Hkv, P, max_pages, num_pages;
    float eps;
    RopeFreqs freqs;
};

template <bool kInt8>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) prologue_kernel(const PrologueParams p)
{
    // Everything this kernel reads may come from the kernel before it, and
    // what it writes may still be read there: wait before touching memory.
    allow_dependent_launch();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    // item = ((b * M + i) * (Hq + Hkv) + head): token i of sequence b sits at
    // position T_b - M + i
    const int heads = p.Hq + p.Hkv;
    const int item = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (item >= p.B * p.M * heads)
        return;
    const int tok = item / heads; // b * M + i
    const int b = tok / p.M;
    const int hh = item % heads;
    const int T = p.context_lens[b];
    if (T < p.M || T > p.max_pages * p.P) {
        if (hh == 0 && tok % p.M == 0 && lane == 0)
            atomicOr(&g_flags_prologue, PGQA_DEVERR_BAD_CONTEXT);
        return;
    }
    const int pos = T - p.M + tok % p.M;
    const bool is_q = hh < p.Hq;
    const int h = is_q ? hh : hh - p.Hq;

    const uint16_t *src;
    const uint16_t *gamma;
    uint16_t *dst = nullptr;
    size_t slot = 0;
    if (is_q) {
        src = p.q + (static_cast<size_t>(tok) * p.Hq + h) * kHeadDim;
        gamma = p.gamma_q;
        dst = p.q_out + (static_cast<size_t>(tok) * p.Hq + h) * kHeadDim;
    } else {
        const int phys = p.block_table[static_cast<size_t>(b) * p.max_pages + pos / p.P];
        if (phys < 0 || phys >= p.num_pages) {
            if (lane == 0)
                atomicOr(&g_flags_prologue, PGQA_DEVERR_BAD_PAGE);
            return;
        }
        slot = ((static_cast<size_t>(phys) * p.Hkv + h) * p.P + pos % p.P) * kHeadDim;
        src = p.k + (static_cast<size_t>(tok) * p.Hkv + h) * kHeadDim;
        gamma = p.gamma_k;
        const uint16_t *vsrc = p.v + (static_cast<size_t>(tok) * p.Hkv + h) * kHeadDim;
        if constexpr (kInt8) {
            float xv[4];
            load_head(vsrc, xv);
            store_row_int8(xv, p.v_cache8 + slot, p.v_scale + slot / kHeadDim);
        } else {
            dst = p.k_cache + slot;
            // V is appended bit for bit: 32 lanes x 8 bytes = one 256-byte row.
            const uint2 *vrow = reinterpret_cast<const uint2 *>(vsrc);
            reinterpret_cast<uint2 *>(p.v_cache + slot)[lane] = vrow[lane];
        }
    }

    float x[4];
    norm_rope_head(src, gamma, p.eps, pos, p.freqs, x);
    if (kInt8 && !is_q) {
        round_head_bf16(x);
        store_row_int8(x, p.k_cache8 + slot, p.k_scale + slot / kHeadDim);
        return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        dst[lane + 32 * i] = f32_to_bf16_bits(x[i]);
}

} // namespace

cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t stream)
{
    if (a.B == 0)
        return cudaSuccess;
    PrologueParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.gamma_q = a.gamma_q;
    p.gamma_k = a.gamma_k;
    p.context_lens = a.context_lens;
    p.block_table = a.block_table;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.q_out = a.q_out;
    p.B = a.B;
    p.M = a.M > 0 ? a.M : 1;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.P = a.page_size;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.eps = a.eps;
    p.freqs = make_rope_freqs(a.rope_theta);
    p.k_cache8 = a.k_cache8;
    p.v_cache8 = a.v_cache8;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    const long items = static_cast<long>(a.B) * p.M * (a.Hq + a.Hkv);
    const unsigned blocks = static_cast<unsigned>((items + kWarpsPerBlock - 1) / kWarpsPerBlock);
    if (a.k_cache8)
        return launch_pdl(prologue_kernel<true>, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, stream, p);
    return launch_pdl(prologue_kernel<false>, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, stream, p);
}

cudaError_t read_flags_prologue(unsigned *flags, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_flags_prologue, sizeof(unsigned));
    if (err == cudaSuccess && clear) {
        const unsigned zero = 0;
        err = cudaMemcpyToSymbol(g_flags_prologue, &zero, sizeof(unsigned));
    }
    return err;
}

} // namespace pgqa
