// tiled.cu -- host-tiled decode attention: the softmax state (m, l, acc)
// lives in global memory across KV tiles copied in from pinned host memory.
//
// "EdgeTransformerEngine", KV-offload design: registers and shared memory
// vanish when a kernel ends, so a state that must survive many tiles is kept
// in global memory and the work is split into three kernels -- init
// (m = -1e30, l = 0, acc = 0), a per-tile update that rescales the state in
// place, and finalize (out = acc / l). Tiles hold 512 positions.
//
// The update kernel runs one thread-block cluster of kTileSplit CTAs per
// (sequence, KV head), each CTA with 8 warps folding a contiguous share of
// the tile's 16-key chunks straight from the (L2-resident, just copied) tile
// with 16-byte loads. Each CTA merges its warps' states in shared memory;
// then CTA 0 of the cluster reads the other CTAs' states through distributed
// shared memory and merges them into the global state. m is stored in
// natural-log units.
#include <algorithm>

#include <cooperative_groups.h>

#include "attn_core.cuh"
#include "launch.h"

namespace pgqa {
namespace {

constexpr int kTileWarps = 8;
constexpr int kTileSplit = 8; // CTAs (one cluster) per (sequence, KV head) and tile

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
    int n_pos, seq_stride, Hq, Hkv;
    float scale_log2;
    float *m, *l, *acc;
};

template <int G>
__global__ void __cluster_dims__(kTileSplit, 1, 1) __launch_bounds__(kTileWarps * 32)
    tile_update_kernel(const TileParams p)
{
    constexpr int kRec = record_floats<G>();
    constexpr int kPerThread = (G * kHeadDim + kTileWarps * 32 - 1) / (kTileWarps * 32);
    __shared__ __align__(16) float recs[kTileWarps][kRec];
    __shared__ __align__(16) float cta_rec[kRec]; // this CTA's state, read by CTA 0 of the cluster
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int warp = threadIdx.x >> 5;
    const int rank = blockIdx.x; // the cluster spans gridDim.x = kTileSplit
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;

    allow_dependent_launch();
    grid_dependency_wait();
    WarpAttn<G> st;
    st.init(p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * kHeadDim, p.scale_log2);
    const long stride = static_cast<long>(p.Hkv) * kRowBytes; // one position, all KV heads
    const size_t base = (static_cast<size_t>(b) * p.seq_stride * p.Hkv + kvh) * kRowBytes;
    const int n_chunks = (p.n_pos + kChunkTokens - 1) / kChunkTokens;
    const int per_cta = (n_chunks + kTileSplit - 1) / kTileSplit;
    const int c_end = min(n_chunks, (rank + 1) * per_cta);
    for (int c = rank * per_cta + warp; c < c_end; c += kTileWarps) {
        const size_t off = base + static_cast<size_t>(c) * kChunkTokens * stride;
        st.fold_chunk(GlobalRows{p.k_tile + off, p.v_tile + off, stride},
                      min(kChunkTokens, p.n_pos - c * kChunkTokens));
    }
    st.reduce_groups();
    st.store_record(recs[warp]);
    __syncthreads();

    // this CTA's state (base-2 m; warps without chunks hold m = -1e30, l = 0)
    for (int e = threadIdx.x; e < G * kHeadDim; e += kTileWarps * 32) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float M = kEmptyMax;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w)
            M = fmaxf(M, recs[w][G * kHeadDim + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w) {
            const float wt = exp2f(recs[w][G * kHeadDim + h] - M);
            L = fmaf(recs[w][G * kHeadDim + G + h], wt, L);
            O = fmaf(recs[w][h * kHeadDim + d], wt, O);
        }
        cta_rec[h * kHeadDim + d] = O;
        if (d == 0) {
            cta_rec[G * kHeadDim + h] = M;
            cta_rec[G * kHeadDim + G + h] = L;
        }
    }
    cluster.sync(); // every CTA's state is complete and visible to the cluster

    if (rank == 0) {
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
            for (int r = 0; r < kTileSplit; ++r)
                M = fmaxf(M, cluster.map_shared_rank(cta_rec, r)[G * kHeadDim + h]);
            const float w_old = exp2f(m_old - M);
            float L = p.l[row] * w_old;
            float O = p.acc[row * kHeadDim + d] * w_old;
#pragma unroll
            for (int r = 0; r < kTileSplit; ++r) {
                const float *rec = cluster.map_shared_rank(cta_rec, r);
                const float wt = exp2f(rec[G * kHeadDim + h] - M);
                L = fmaf(rec[G * kHeadDim + G + h], wt, L);
                O = fmaf(rec[h * kHeadDim + d], wt, O);
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
    cluster.sync(); // the other CTAs keep their state until CTA 0 has read it
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

// Zero-copy variant: the whole history [B][T][Hkv][128] stays in pinned host
// memory mapped into the device address space, and the kernel reads it over
// the host link directly (no device copy of the tiles). Grid (partition, KV
// head, sequence): each CTA folds positions [part * len, part * len + len)
// with 8 warps as in the tile update, merges its warps in shared memory and
// writes the output (one partition) or its partition state (m in natural-log
// units) for merge_kernel.
struct DirectParams {
    const __nv_bfloat16 *q;
    const char *k, *v;
    int T, len, NP, Hq, Hkv;
    float scale_log2;
    float *out_f32;
    uint16_t *out_bf16;
    float *ws_m, *ws_l, *ws_acc;
};

template <int G>
__global__ void __launch_bounds__(kTileWarps * 32) host_direct_kernel(const DirectParams p)
{
    constexpr int kRec = record_floats<G>();
    __shared__ __align__(16) float recs[kTileWarps][kRec];
    const int warp = threadIdx.x >> 5;
    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

    allow_dependent_launch();
    grid_dependency_wait();
    WarpAttn<G> st;
    st.init(p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * kHeadDim, p.scale_log2);
    const int p0 = part * p.len;
    const int n_pos = max(0, min(p.T - p0, p.len));
    const long stride = static_cast<long>(p.Hkv) * kRowBytes; // one position, all KV heads
    const size_t base = ((static_cast<size_t>(b) * p.T + p0) * p.Hkv + kvh) * kRowBytes;
    const int n_chunks = (n_pos + kChunkTokens - 1) / kChunkTokens;
    for (int c = warp; c < n_chunks; c += kTileWarps) {
        const size_t off = base + static_cast<size_t>(c) * kChunkTokens * stride;
        st.fold_chunk(GlobalRows{p.k + off, p.v + off, stride},
                      min(kChunkTokens, n_pos - c * kChunkTokens));
    }
    st.reduce_groups();
    st.store_record(recs[warp]);
    __syncthreads();

    for (int e = threadIdx.x; e < G * kHeadDim; e += kTileWarps * 32) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float M = kEmptyMax;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w)
            M = fmaxf(M, recs[w][G * kHeadDim + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kTileWarps; ++w) {
            const float wt = exp2f(recs[w][G * kHeadDim + h] - M);
            L = fmaf(recs[w][G * kHeadDim + G + h], wt, L);
            O = fmaf(recs[w][h * kHeadDim + d], wt, O);
        }
        const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + h;
        if (p.NP == 1) {
            const float o = L > 0.f ? O / L : 0.f;
            if (p.out_f32)
                p.out_f32[row * kHeadDim + d] = o;
            if (p.out_bf16)
                p.out_bf16[row * kHeadDim + d] = f32_to_bf16_bits(o);
        } else {
            const size_t idx = row * p.NP + part;
            if (d == 0) {
                p.ws_m[idx] = M * kLn2; // natural-log units, as attn_partition_merge takes them
                p.ws_l[idx] = L;
            }
            p.ws_acc[idx * kHeadDim + d] = O;
        }
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
    p.seq_stride = a.seq_stride > 0 ? a.seq_stride : a.n_pos;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.scale_log2 = a.scale * kLog2e;
    p.m = a.m;
    p.l = a.l;
    p.acc = a.acc;
    const dim3 grid(kTileSplit, a.Hkv, a.B);
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

int host_direct_partitions(int B, int Hkv, int T, int requested, int sm_count)
{
    if (T <= 0)
        return 1;
    const long max_np = (T + kHostDirectMinPositions - 1) / kHostDirectMinPositions;
    long np = requested;
    if (np <= 0) {
        // one wave of CTAs: the link, not the SMs, bounds the stream
        const long units = static_cast<long>(B) * Hkv;
        const long slots = sm_count > 0 ? sm_count : 1;
        np = std::max<long>(1, slots / std::max<long>(1, units));
        np = std::min(np, max_np);
    }
    np = std::min<long>(std::max<long>(np, 1), std::min<long>(T, kMaxPartitions));
    const long len = (T + np - 1) / np;
    return static_cast<int>((T + len - 1) / len);
}

size_t host_direct_workspace_bytes(int B, int Hq, int num_partitions)
{
    if (num_partitions <= 1)
        return 0;
    const size_t n = static_cast<size_t>(B) * Hq * num_partitions;
    const auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    return 2 * a256(n * sizeof(float)) + a256(n * kHeadDim * sizeof(float));
}

cudaError_t launch_host_direct(const HostDirectArgs &a, cudaStream_t stream)
{
    if (a.B == 0)
        return cudaSuccess;
    DirectParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    p.k = reinterpret_cast<const char *>(a.k);
    p.v = reinterpret_cast<const char *>(a.v);
    p.T = a.T;
    p.NP = a.num_partitions;
    p.len = a.T > 0 ? (a.T + a.num_partitions - 1) / a.num_partitions : 0;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.scale_log2 = a.scale * kLog2e;
    p.out_f32 = a.out_f32;
    p.out_bf16 = reinterpret_cast<uint16_t *>(a.out_bf16);
    if (a.num_partitions > 1) {
        const size_t n = static_cast<size_t>(a.B) * a.Hq * a.num_partitions;
        const auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
        char *ws = reinterpret_cast<char *>(a.ws);
        p.ws_m = reinterpret_cast<float *>(ws);
        p.ws_l = reinterpret_cast<float *>(ws + a256(n * sizeof(float)));
        p.ws_acc = reinterpret_cast<float *>(ws + 2 * a256(n * sizeof(float)));
    }
    const dim3 grid(a.num_partitions, a.Hkv, a.B);
    const dim3 block(kTileWarps * 32);
    cudaError_t err;
    switch (a.Hq / a.Hkv) {
    case 1: err = launch_pdl(host_direct_kernel<1>, grid, block, 0, stream, p); break;
    case 2: err = launch_pdl(host_direct_kernel<2>, grid, block, 0, stream, p); break;
    case 3: err = launch_pdl(host_direct_kernel<3>, grid, block, 0, stream, p); break;
    case 4: err = launch_pdl(host_direct_kernel<4>, grid, block, 0, stream, p); break;
    case 5: err = launch_pdl(host_direct_kernel<5>, grid, block, 0, stream, p); break;
    case 6: err = launch_pdl(host_direct_kernel<6>, grid, block, 0, stream, p); break;
    case 7: err = launch_pdl(host_direct_kernel<7>, grid, block, 0, stream, p); break;
    case 8: err = launch_pdl(host_direct_kernel<8>, grid, block, 0, stream, p); break;
    default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess || a.num_partitions <= 1)
        return err;
    MergeArgs ma{};
    ma.m = p.ws_m;
    ma.l = p.ws_l;
    ma.acc = p.ws_acc;
    ma.B = a.B;
    ma.Hq = a.Hq;
    ma.NP = a.num_partitions;
    ma.out_f32 = a.out_f32;
    ma.out_bf16 = a.out_bf16;
    return launch_merge(ma, stream);
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
