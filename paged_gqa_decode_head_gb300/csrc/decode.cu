// decode.cu -- paged GQA decode attention, split over KV partitions, and the
// exact partition merge.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime":
//   s10.1 one CTA per (sequence, KV head) serves all g query heads of the
//         group, so every K/V byte is read from HBM once;
//   s10.2 the history is cut into partitions, one CTA each, whose
//         (m_p, l_p, o_p) go to a preallocated fp32 scratch, and a second
//         launch merges them;
//   s9.1  the merge rescales every partition to the common maximum, which is
//         exact (not an approximation);
//   s12.1 / s12.2 multi-stage prefetch, 16-byte aligned copies, masked tails.
//
// GB300 design. Grid = (partition, KV head, sequence). Each of the CTA's 4
// warps owns every 4th 16-key chunk of the partition and a private ring of 3
// shared-memory stages; lane 0 of the warp looks the chunk's physical page up
// in the block table and issues two 4 KiB bulk TMA copies (K rows, V rows:
// the rows of one page and KV head are contiguous) that complete on the
// stage's mbarrier. The warp folds each staged chunk into its (m, l, acc)
// (attn_core.cuh) and refills the stage with the chunk 3 ahead. At the end the
// warps' states are merged through shared memory; NP = 1 writes the output,
// NP > 1 writes the partition state and the merge kernel finishes.
#include <algorithm>
#include <cmath>

#include "attn_core.cuh"
#include "launch.h"

namespace pgqa {
namespace {

__device__ unsigned g_flags_decode;

__device__ __forceinline__ void raise_flag(unsigned f) { atomicOr(&g_flags_decode, f); }

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kChunkBytes; // K chunk then V chunk
constexpr int kCtasPerSm = 2;                // what the shared-memory footprint allows
constexpr int kSplitSmem = kWarps * kStages * kStageBytes + kWarps * kStages * 8;

struct SplitParams {
    const __nv_bfloat16 *q;
    const char *k_cache, *v_cache;
    const int32_t *block_table, *context_lens;
    float *out_f32;
    uint16_t *out_bf16;
    float *ws_m, *ws_l, *ws_acc;
    int Hq, Hkv, P, max_pages, num_pages, NP, ppp;
    float scale_log2;
};

template <int G>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const SplitParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;

    int T = p.context_lens[b];
    if (T < 0 || T > p.max_pages * p.P) {
        if (part == 0 && threadIdx.x == 0)
            raise_flag(PGQA_DEVERR_BAD_CONTEXT);
        T = 0;
    }
    const int part_tokens = p.ppp * p.P;
    const int n_parts = max(1, (T + part_tokens - 1) / part_tokens);
    if (part >= n_parts)
        return; // this sequence is shorter than the launch's longest
    const int tok0 = part * part_tokens;
    const int tok1 = min(T, tok0 + part_tokens);
    const int n_chunks = max(0, (tok1 - tok0 + kChunkTokens - 1) / kChunkTokens);
    const int my_chunks = (n_chunks > warp) ? (n_chunks - 1 - warp) / kWarps + 1 : 0;

    unsigned char *stages = smem + warp * kStages * kStageBytes;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + kWarps * kStages * kStageBytes) + warp * kStages;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int32_t *table = p.block_table + static_cast<size_t>(b) * p.max_pages;
    // k-th chunk of this warp starts at token tok0 + (warp + k*kWarps)*16, which
    // never straddles a page because page_size is a multiple of 16.
    auto chunk_token = [&](int k) { return tok0 + (warp + k * kWarps) * kChunkTokens; };
    auto issue = [&](int k, uint64_t policy) {
        const int t = chunk_token(k);
        const int phys = table[t / p.P];
        uint64_t *bar = &bars[k % kStages];
        if (phys < 0 || phys >= p.num_pages) {
            raise_flag(PGQA_DEVERR_BAD_PAGE);
            mbar_arrive(bar); // complete the phase with no data; the keys are masked
            return;
        }
        const size_t row0 = (static_cast<size_t>(phys) * p.Hkv + kvh) * p.P + (t % p.P);
        unsigned char *dst = stages + (k % kStages) * kStageBytes;
        mbar_arrive_expect_tx(bar, kStageBytes);
        bulk_copy_g2s(dst, p.k_cache + row0 * kRowBytes, kChunkBytes, bar, policy);
        bulk_copy_g2s(dst + kChunkBytes, p.v_cache + row0 * kRowBytes, kChunkBytes, bar, policy);
    };

    uint64_t policy = 0;
    if (lane == 0) {
        policy = l2_evict_first_policy();
        const int first = min(kStages, my_chunks);
        for (int k = 0; k < first; ++k)
            issue(k, policy);
    }

    WarpAttn<G> st;
    st.init(p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * kHeadDim, p.scale_log2);

    int k = 0;
    bool ok = true;
    for (; k < my_chunks; ++k) {
        const int s = k % kStages;
        const bool landed = mbar_wait_bounded(&bars[s], (k / kStages) & 1);
        if (!__all_sync(0xFFFFFFFFu, landed)) { // keep the warp's lanes in step
            ok = false;
            break;
        }
        const int t = chunk_token(k);
        const int phys = table[t / p.P];
        const int n_valid = (phys >= 0 && phys < p.num_pages) ? min(kChunkTokens, tok1 - t) : 0;
        const uint32_t a = smem_addr(stages + s * kStageBytes);
        st.fold_chunk(SmemRows{a, a + kChunkBytes}, n_valid);
        __syncwarp();
        if (lane == 0 && k + kStages < my_chunks) {
            fence_proxy_async_smem();
            issue(k + kStages, policy);
        }
    }
    if (!ok) {
        // A copy never completed: flag it, wait (bounded) for the copies
        // still in flight into this warp's stages, and contribute nothing.
        if (lane == 0)
            raise_flag(PGQA_DEVERR_WAIT_TIMEOUT);
        const int issued = min(my_chunks, k + kStages);
        for (int kk = k; kk < issued; ++kk)
            (void)mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            st.m[h] = kEmptyMax;
            st.l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < WarpAttn<G>::DPL; ++e)
                st.acc[h][e] = 0.f;
        }
    }

    st.reduce_groups();
    __syncwarp();
    // Every copy into this warp's stages has landed, so the stages can hold
    // the warp's state record.
    st.store_record(reinterpret_cast<float *>(stages));
    __syncthreads();

    const int base_q = kvh * G;
    for (int e = threadIdx.x; e < G * kHeadDim; e += kWarps * 32) {
        const int h = e / kHeadDim;
        const int d = e % kHeadDim;
        float M = kEmptyMax;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * kStages * kStageBytes);
            M = fmaxf(M, rec[G * kHeadDim + h]);
        }
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * kStages * kStageBytes);
            const float wt = exp2f(rec[G * kHeadDim + h] - M);
            L = fmaf(rec[G * kHeadDim + G + h], wt, L);
            O = fmaf(rec[h * kHeadDim + d], wt, O);
        }
        const size_t row = static_cast<size_t>(b) * p.Hq + base_q + h;
        if (n_parts == 1) {
            const float o = L > 0.f ? O / L : 0.f;
            if (p.out_f32)
                p.out_f32[row * kHeadDim + d] = o;
            if (p.out_bf16)
                p.out_bf16[row * kHeadDim + d] = f32_to_bf16_bits(o);
        } else {
            const size_t idx = row * p.NP + part;
            if (d == 0) {
                p.ws_m[idx] = M; // base-2 units (private workspace format)
                p.ws_l[idx] = L;
            }
            p.ws_acc[idx * kHeadDim + d] = O;
        }
    }
}

struct MergeParams {
    const float *m, *l, *acc;
    int Hq, NP;
    float *out_f32;
    uint16_t *out_bf16;
    const int32_t *context_lens;
    int P, ppp, max_pages;
};

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// One CTA per (sequence, query head). Pass 1 finds M = max_p m_p; pass 2 has
// warp w accumulate partitions w, w+8, ... with lane i owning dims 4i..4i+3;
// the 8 warps' sums are then combined in shared memory.
template <bool kBase2>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p)
{
    __shared__ float red_max[kMergeWarps];
    __shared__ float red_l[kMergeWarps];
    __shared__ float4 red_o[kMergeWarps][32];
    const int row = blockIdx.x; // b * Hq + h
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int np = p.NP;
    if (p.context_lens) {
        const int b = row / p.Hq;
        int T = p.context_lens[b];
        if (T < 0 || T > p.max_pages * p.P)
            T = 0;
        const int part_tokens = p.ppp * p.P;
        np = min(np, max(1, (T + part_tokens - 1) / part_tokens));
        if (np == 1)
            return; // a single partition wrote this sequence's output itself
    }
    const float *m = p.m + static_cast<size_t>(row) * p.NP;
    const float *l = p.l + static_cast<size_t>(row) * p.NP;
    const float4 *acc = reinterpret_cast<const float4 *>(p.acc + static_cast<size_t>(row) * p.NP * kHeadDim);

    float M = -INFINITY;
    for (int i = threadIdx.x; i < np; i += kMergeThreads)
        M = fmaxf(M, __ldcg(m + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    if (lane == 0)
        red_max[warp] = M;
    __syncthreads();
    M = red_max[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w)
        M = fmaxf(M, red_max[w]);
    if (M == -INFINITY)
        M = 0.f; // every m is -inf: all weights become 0

    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int i = warp; i < np; i += kMergeWarps) {
        const float mi = __ldcg(m + i);
        const float wt = kBase2 ? exp2f(mi - M) : expf(mi - M);
        L = fmaf(__ldcg(l + i), wt, L);
        const float4 a = __ldcg(acc + static_cast<size_t>(i) * (kHeadDim / 4) + lane);
        o.x = fmaf(a.x, wt, o.x);
        o.y = fmaf(a.y, wt, o.y);
        o.z = fmaf(a.z, wt, o.z);
        o.w = fmaf(a.w, wt, o.w);
    }
    red_o[warp][lane] = o;
    if (lane == 0)
        red_l[warp] = L;
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
        const int d = threadIdx.x;
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            Ls += red_l[w];
            Os += reinterpret_cast<const float *>(&red_o[w][0])[d];
        }
        const float out = Ls > 0.f ? Os / Ls : 0.f;
        if (p.out_f32)
            p.out_f32[static_cast<size_t>(row) * kHeadDim + d] = out;
        if (p.out_bf16)
            p.out_bf16[static_cast<size_t>(row) * kHeadDim + d] = f32_to_bf16_bits(out);
    }
}

constexpr int kMaxDevices = 64;

template <int G> cudaError_t launch_split(const SplitParams &kp, dim3 grid, cudaStream_t stream)
{
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= kMaxDevices || !configured[dev]) {
        err = cudaFuncSetAttribute(decode_split_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kSplitSmem);
        if (err != cudaSuccess)
            return err;
        if (dev < kMaxDevices)
            configured[dev] = true;
    }
    decode_split_kernel<G><<<grid, kWarps * 32, kSplitSmem, stream>>>(kp);
    return cudaGetLastError();
}

} // namespace

int choose_partitions(int B, int Hkv, int page_size, int max_pages, int requested, int sm_count)
{
    if (max_pages <= 0)
        return 1;
    long np;
    if (requested > 0) {
        np = requested;
    } else {
        // Fill every CTA slot of one wave, keep partitions between 128 and
        // 1024 positions (long enough to amortise the merge, short enough to
        // balance ragged batches).
        const long units = static_cast<long>(B) * Hkv;
        const long slots = static_cast<long>(sm_count > 0 ? sm_count : 1) * kCtasPerSm;
        long ppp = (units * max_pages + slots - 1) / slots;
        const long lo = std::max(1, 128 / page_size);
        const long hi = std::max(1, 1024 / page_size);
        ppp = std::min(std::max(ppp, lo), hi);
        np = (max_pages + ppp - 1) / ppp;
    }
    np = std::min<long>(std::max<long>(np, 1), std::min(max_pages, kMaxPartitions));
    const long ppp = (max_pages + np - 1) / np;
    return static_cast<int>((max_pages + ppp - 1) / ppp);
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t decode_workspace_bytes(int B, int Hq, int num_partitions)
{
    if (num_partitions <= 1)
        return 0;
    const size_t n = static_cast<size_t>(B) * Hq * num_partitions;
    return 2 * align256(n * sizeof(float)) + align256(n * kHeadDim * sizeof(float));
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream)
{
    const int G = a.Hq / a.Hkv;
    SplitParams kp{};
    kp.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    kp.k_cache = reinterpret_cast<const char *>(a.k_cache);
    kp.v_cache = reinterpret_cast<const char *>(a.v_cache);
    kp.block_table = a.block_table;
    kp.context_lens = a.context_lens;
    kp.out_f32 = a.out_f32;
    kp.out_bf16 = a.out_bf16;
    kp.Hq = a.Hq;
    kp.Hkv = a.Hkv;
    kp.P = a.page_size;
    kp.max_pages = a.max_pages;
    kp.num_pages = a.num_pages;
    kp.NP = a.num_partitions;
    kp.ppp = a.pages_per_part;
    kp.scale_log2 = a.scale * kLog2e;
    if (a.num_partitions > 1) {
        const size_t n = static_cast<size_t>(a.B) * a.Hq * a.num_partitions;
        char *ws = reinterpret_cast<char *>(a.ws);
        kp.ws_m = reinterpret_cast<float *>(ws);
        kp.ws_l = reinterpret_cast<float *>(ws + align256(n * sizeof(float)));
        kp.ws_acc = reinterpret_cast<float *>(ws + 2 * align256(n * sizeof(float)));
    }
    const dim3 grid(a.num_partitions, a.Hkv, a.B);
    cudaError_t err;
    switch (G) {
    case 1: err = launch_split<1>(kp, grid, stream); break;
    case 2: err = launch_split<2>(kp, grid, stream); break;
    case 3: err = launch_split<3>(kp, grid, stream); break;
    case 4: err = launch_split<4>(kp, grid, stream); break;
    case 5: err = launch_split<5>(kp, grid, stream); break;
    case 6: err = launch_split<6>(kp, grid, stream); break;
    case 7: err = launch_split<7>(kp, grid, stream); break;
    case 8: err = launch_split<8>(kp, grid, stream); break;
    default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess || a.num_partitions <= 1)
        return err;
    MergeArgs ma{};
    ma.m = kp.ws_m;
    ma.l = kp.ws_l;
    ma.acc = kp.ws_acc;
    ma.B = a.B;
    ma.Hq = a.Hq;
    ma.NP = a.num_partitions;
    ma.out_f32 = a.out_f32;
    ma.out_bf16 = a.out_bf16;
    ma.context_lens = a.context_lens;
    ma.page_size = a.page_size;
    ma.pages_per_part = a.pages_per_part;
    ma.max_pages = a.max_pages;
    return launch_merge(ma, stream);
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t stream)
{
    if (a.B == 0 || a.Hq == 0)
        return cudaSuccess;
    MergeParams mp{};
    mp.m = a.m;
    mp.l = a.l;
    mp.acc = a.acc;
    mp.Hq = a.Hq;
    mp.NP = a.NP;
    mp.out_f32 = a.out_f32;
    mp.out_bf16 = reinterpret_cast<uint16_t *>(a.out_bf16);
    mp.context_lens = a.context_lens;
    mp.P = a.page_size;
    mp.ppp = a.pages_per_part;
    mp.max_pages = a.max_pages;
    const unsigned rows = static_cast<unsigned>(a.B) * a.Hq;
    if (a.context_lens)
        merge_kernel<true><<<rows, kMergeThreads, 0, stream>>>(mp);
    else
        merge_kernel<false><<<rows, kMergeThreads, 0, stream>>>(mp);
    return cudaGetLastError();
}

cudaError_t read_flags_decode(unsigned *flags, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_flags_decode, sizeof(unsigned));
    if (err == cudaSuccess && clear) {
        const unsigned zero = 0;
        err = cudaMemcpyToSymbol(g_flags_decode, &zero, sizeof(unsigned));
    }
    return err;
}

} // namespace pgqa
