// tiled.cu -- host-tiled decode attention: the softmax state (m, l, acc)
// lives in global memory across KV tiles copied in from pinned host memory.
//
// "EdgeTransformerEngine", KV-offload design: registers and shared memory
// vanish when a kernel ends, so a state that must survive many tiles is kept
// in global memory and the work is split into three kernels -- init
// (m = -1e30, l = 0, acc = 0), a per-tile update that rescales the state in
// place, and finalize (out = acc / l). Tiles hold 512 positions.
//
// The update kernel runs one CTA per (sequence, KV head) with 8 warps; each
// warp folds 16-key chunks straight from the (L2-resident, just copied) tile
// with 16-byte loads, the warps' states are merged in shared memory, and the
// result is merged into the global state. m is stored in natural-log units.
#include "attn_core.cuh"
#include "launch.h"

namespace pgqa {
namespace {

constexpr int kTileWarps = 8;

__global__ void tile_init_kernel(float *m, float *l, float *acc, int rows)
{
    allow_dependent_launch();
    grid_dependency_wait();
    const long n = static_cast<long>(rows) * kHeadDim;
    for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long>(gridDim.x) * blockDim.x) {
        acc[i] = 0.f;
        if (i < rows) {
            m[i] = kEmptyMax;
            l[i] = 0.f;
        }
    }
}

struct TileParams {
    const __nv_bfloat16 *q;
    const char *k_tile, *v_tile;
    int n_pos, Hq, Hkv;
    float scale_log2;
    float *m, *l, *acc;
};

template <int G>
__global__ void __launch_bounds__(kTileWarps * 32) tile_update_kernel(const TileParams p)
{
    constexpr int kRec = record_floats<G>();
    constexpr int kPerThread = (G * kHeadDim + kTileWarps * 32 - 1) / (kTileWarps * 32);
    __shared__ __align__(16) float recs[kTileWarps][kRec];
    const int warp = threadIdx.x >> 5;
    const int kvh = blockIdx.x;
    const int b = blockIdx.y;

    allow_dependent_launch();
    grid_dependency_wait();
    WarpAttn<G> st;
    st.init(p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * kHeadDim, p.scale_log2);
    const long stride = static_cast<long>(p.Hkv) * kRowBytes; // one position, all KV heads
    const size_t base = (static_cast<size_t>(b) * p.n_pos * p.Hkv + kvh) * kRowBytes;
    const int n_chunks = (p.n_pos + kChunkTokens - 1) / kChunkTokens;
    for (int c = warp; c < n_chunks; c += kTileWarps) {
        const size_t off = base + static_cast<size_t>(c) * kChunkTokens * stride;
        st.fold_chunk(GlobalRows{p.k_tile + off, p.v_tile + off, stride},
                      min(kChunkTokens, p.n_pos - c * kChunkTokens));
    }
    st.reduce_groups();
    st.store_record(recs[warp]);
    __syncthreads();

    float newM[kPerThread], newL[kPerThread], newO[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int e = threadIdx.x + i * kTileWarps * 32;
        if (e >= G * kHeadDim)
            break;
        const int h = e / kHeadDim, d = e % kHeadDim;
        const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + h;
        const float m_old = p.m[row] * kLog2e;
        float M = m_old;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w)
            M = fmaxf(M, recs[w][G * kHeadDim + h]);
        const float w_old = exp2f(m_old - M);
        float L = p.l[row] * w_old;
        float O = p.acc[row * kHeadDim + d] * w_old;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w) {
            const float wt = exp2f(recs[w][G * kHeadDim + h] - M);
            L = fmaf(recs[w][G * kHeadDim + G + h], wt, L);
            O = fmaf(recs[w][h * kHeadDim + d], wt, O);
        }
        newM[i] = M, newL[i] = L, newO[i] = O;
    }
    __syncthreads(); // every thread has read the old (m, l) before any is replaced
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int e = threadIdx.x + i * kTileWarps * 32;
        if (e >= G * kHeadDim)
            break;
        const int h = e / kHeadDim, d = e % kHeadDim;
        const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + h;
        p.acc[row * kHeadDim + d] = newO[i];
        if (d == 0) {
            p.m[row] = newM[i] * kLn2;
            p.l[row] = newL[i];
        }
    }
}

__global__ void tile_finalize_kernel(const float *l, const float *acc, int rows, float *out_f32,
                                     uint16_t *out_bf16)
{
    allow_dependent_launch();
    grid_dependency_wait();
    const long n = static_cast<long>(rows) * kHeadDim;
    for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long>(gridDim.x) * blockDim.x) {
        const float den = l[i / kHeadDim];
        const float o = den > 0.f ? acc[i] / den : 0.f;
        if (out_f32)
            out_f32[i] = o;
        if (out_bf16)
            out_bf16[i] = f32_to_bf16_bits(o);
    }
}

unsigned elementwise_blocks(long n)
{
    const long b = (n + 255) / 256;
    return static_cast<unsigned>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

} // namespace

cudaError_t launch_tile_init(float *m, float *l, float *acc, int B, int Hq, cudaStream_t stream)
{
    const int rows = B * Hq;
    if (rows == 0)
        return cudaSuccess;
    return launch_pdl(tile_init_kernel, dim3(elementwise_blocks(static_cast<long>(rows) * kHeadDim)),
                      dim3(256), 0, stream, m, l, acc, rows);
}

cudaError_t launch_tile_update(const TileArgs &a, cudaStream_t stream)
{
    if (a.B == 0 || a.n_pos == 0)
        return cudaSuccess;
    TileParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    p.k_tile = reinterpret_cast<const char *>(a.k_tile);
    p.v_tile = reinterpret_cast<const char *>(a.v_tile);
    p.n_pos = a.n_pos;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.scale_log2 = a.scale * kLog2e;
    p.m = a.m;
    p.l = a.l;
    p.acc = a.acc;
    const dim3 grid(a.Hkv, a.B);
    const int threads = kTileWarps * 32;
    const dim3 block(threads);
    switch (a.Hq / a.Hkv) {
    case 1: return launch_pdl(tile_update_kernel<1>, grid, block, 0, stream, p);
    case 2: return launch_pdl(tile_update_kernel<2>, grid, block, 0, stream, p);
    case 3: return launch_pdl(tile_update_kernel<3>, grid, block, 0, stream, p);
    case 4: return launch_pdl(tile_update_kernel<4>, grid, block, 0, stream, p);
    case 5: return launch_pdl(tile_update_kernel<5>, grid, block, 0, stream, p);
    case 6: return launch_pdl(tile_update_kernel<6>, grid, block, 0, stream, p);
    case 7: return launch_pdl(tile_update_kernel<7>, grid, block, 0, stream, p);
    case 8: return launch_pdl(tile_update_kernel<8>, grid, block, 0, stream, p);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tile_finalize(const float *m, const float *l, const float *acc, int B, int Hq,
                                 float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream)
{
    (void)m;
    const int rows = B * Hq;
    if (rows == 0)
        return cudaSuccess;
    return launch_pdl(tile_finalize_kernel, dim3(elementwise_blocks(static_cast<long>(rows) * kHeadDim)),
                      dim3(256), 0, stream, l, acc, rows, out_f32, reinterpret_cast<uint16_t *>(out_bf16));
}

} // namespace pgqa
