// partition_merge.cuh -- the merge of a (sequence, KV head)'s partition
// states, run inside the attention kernel by the last of its CTAs to finish.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime" s9.1: partial
// (m, l, acc) states combine exactly, with weights e^(m_p - M) against the
// largest partition maximum M; here m is in base-2 units, so the weights are
// 2^(m_p - M). s10.2 runs this as a second launch; the attention kernels of
// this library run it in the CTA that takes the last ticket, which saves one
// dependent launch per layer.
#pragma once

#include "common.cuh"

namespace pgqa {

// Shared memory the merge needs beyond the G x n accumulators: the weights
// [NCOL][kMaxParts], the per-column sums (16 floats) and a float4 per thread.
template <int kThreads, int kMaxParts> constexpr int merge_scratch_bytes(int max_cols)
{
    return max_cols * kMaxParts * 4 + 64 + kThreads * 16;
}

// Merges the n (2 .. kMaxParts) partition states of NCOL query columns from
// the workspace and writes the normalised outputs, in one round trip to
// memory: the NCOL x n accumulators are bulk-copied into shared memory (one
// copy per column) while one warp per column loads m and l and forms the
// weights 2^(m_p - M) and L with shuffles; then every thread folds its share
// of the accumulators from shared memory.
//
// row_of(c) is the row of column c in the [rows][NP] m / l and
// [rows][NP][128] acc workspace and in the [rows][128] outputs. smem must
// hold NCOL * n * 512 bytes plus merge_scratch_bytes and be free (every
// earlier copy into it landed); bar is a spare mbarrier slot. The caller has
// acquired the other CTAs' stores (its ticket) and ordered them for all its
// threads. Returns false, leaving the outputs alone, if the bulk copy did
// not land within the bounded wait (after a second bounded wait, since the
// copy writes this CTA's shared memory).
template <int NCOL, int kThreads, int kMaxParts, typename RowOf>
__device__ bool merge_partitions_in_cta(const float *ws_m, const float *ws_l, const float *ws_acc, int NP, int n,
                                        RowOf row_of, float *out_f32, uint16_t *out_bf16, unsigned char *smem,
                                        uint64_t *bar)
{
    static_assert(kMaxParts <= 64, "one warp loads at most 64 partition maxima");
    constexpr int kWarpsM = kThreads / 32;
    float *acc = reinterpret_cast<float *>(smem);              // [NCOL][n][128]
    float *w = acc + static_cast<size_t>(NCOL) * n * kHeadDim; // [NCOL][kMaxParts] weights
    float *Ls = w + NCOL * kMaxParts;                          // [NCOL], padded to 16 floats
    float4 *red = reinterpret_cast<float4 *>(Ls + 16);         // [kThreads] partial sums
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // One bulk copy per column. A thread issues them one after another (each
    // takes its issuing thread a fraction of a microsecond), so more than two
    // columns spread over the warps, after a barrier that publishes the
    // mbarrier's initialisation: M = 4 fused step (8 columns) 10.91 -> 10.71
    // us per layer; with 2 columns the barrier costs more than it saves
    // (attention alone 8.71 -> 8.83).
    constexpr bool kSpreadCopies = NCOL > 2;
    const uint32_t row_bytes = static_cast<uint32_t>(n) * kHeadDim * 4;
    const auto copy_column = [&](int h) {
        // the stage area was last used through the generic proxy, and the
        // other CTAs' partition states were acquired through it
        fence_proxy_async_smem();
        fence_proxy_async_global();
        bulk_copy_g2s_nohint(acc + static_cast<size_t>(h) * n * kHeadDim, ws_acc + row_of(h) * NP * kHeadDim,
                             row_bytes, bar);
    };
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, NCOL * row_bytes);
        if constexpr (!kSpreadCopies) {
#pragma unroll
            for (int h = 0; h < NCOL; ++h)
                copy_column(h);
        }
    }
    if constexpr (kSpreadCopies) {
        __syncthreads();
        if (lane == 0)
            for (int h = warp; h < NCOL; h += kWarpsM)
                copy_column(h);
    }
    for (int h = warp; h < NCOL; h += kWarpsM) {
        const float *mh = ws_m + row_of(h) * NP;
        const float *lh = ws_l + row_of(h) * NP;
        const float m0 = lane < n ? __ldcg(mh + lane) : kEmptyMax;
        const float m1 = lane + 32 < n ? __ldcg(mh + lane + 32) : kEmptyMax;
        const float l0 = lane < n ? __ldcg(lh + lane) : 0.f;
        const float l1 = lane + 32 < n ? __ldcg(lh + lane + 32) : 0.f;
        float M = fmaxf(m0, m1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
        const float w0 = exp2f(m0 - M), w1 = exp2f(m1 - M);
        float L = l0 * w0 + l1 * w1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            L += __shfl_xor_sync(0xFFFFFFFFu, L, off);
        w[h * kMaxParts + lane] = w0;
        if (lane + 32 < kMaxParts)
            w[h * kMaxParts + lane + 32] = w1;
        if (lane == 0)
            Ls[h] = L;
    }
    __syncthreads();
    if (!mbar_wait_bounded(bar, 0)) {
        (void)mbar_wait_bounded(bar, 0);
        return false;
    }
    constexpr int kItems = NCOL * 32; // (column, 4 dims)
    constexpr int kSlices = kThreads >= kItems ? kThreads / kItems : 1;
    constexpr int kLanesPerSlice = kThreads / kSlices;
    for (int base = 0; base < kItems; base += kLanesPerSlice) {
        const int item = base + (threadIdx.x % kLanesPerSlice);
        const int slice = threadIdx.x / kLanesPerSlice;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        if (item < kItems && slice < kSlices) {
            const int h = item / 32, d4 = item % 32;
            const float4 *src = reinterpret_cast<const float4 *>(acc + static_cast<size_t>(h) * n * kHeadDim) + d4;
            // unrolled so that several partitions' loads are in flight at
            // once (the sum's order is unchanged): M = 4 fused step 11.19 ->
            // 11.09 us per layer
#pragma unroll 4
            for (int part = slice; part < n; part += kSlices) {
                const float4 v = src[static_cast<size_t>(part) * (kHeadDim / 4)];
                const float wt = w[h * kMaxParts + part];
                sum.x = fmaf(v.x, wt, sum.x);
                sum.y = fmaf(v.y, wt, sum.y);
                sum.z = fmaf(v.z, wt, sum.z);
                sum.w = fmaf(v.w, wt, sum.w);
            }
        }
        red[threadIdx.x] = sum;
        __syncthreads();
        if (slice == 0 && item < kItems) {
            for (int sl = 1; sl < kSlices; ++sl) {
                const float4 v = red[threadIdx.x + sl * kLanesPerSlice];
                sum.x += v.x, sum.y += v.y, sum.z += v.z, sum.w += v.w;
            }
            const int h = item / 32, d4 = item % 32;
            const float L = Ls[h];
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float r[4] = {sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv};
            const size_t off = row_of(h) * kHeadDim + 4 * d4;
            if (out_f32)
                *reinterpret_cast<float4 *>(out_f32 + off) = make_float4(r[0], r[1], r[2], r[3]);
            if (out_bf16)
                *reinterpret_cast<uint2 *>(out_bf16 + off) =
                    make_uint2(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]));
        }
        __syncthreads();
    }
    return true;
}

} // namespace pgqa
