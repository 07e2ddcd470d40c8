// attn_core.cuh -- one warp folds 16-key chunks of K/V into the online
// softmax state (m, l, acc) of the g query heads of one KV head.
//
// Math ("EdgeTransformerEngine", online-softmax note; "From Qwen3 math to
// CUDA kernels", s2.6 and s9.1): for each key, newm = max(m, s),
// corr = e^(m - newm), p = e^(s - newm), l = l*corr + p, acc = acc*corr + p*V.
// Here the rescale is applied once per 16-key chunk with the chunk's maximum
// (the same state, reached in fewer rescales), and scores are kept in base-2
// units: q is pre-multiplied by scale*log2(e) so exp2 replaces exp.
//
// Lane layout. LPK lanes share one key (LPK = 8 for g <= 4, 16 for g > 4);
// a warp covers KPP = 32/LPK keys per pass and 16/KPP passes per chunk. Lane
// `sub` (0..LPK-1) of a key owns the 8-dim segments starting at dims
// (j*LPK + sub)*8, j < NSEG, so the LPK lanes of a key read one 16-byte
// vector each from a contiguous stretch of the row (conflict-free shared
// loads, coalesced global loads). Partial dot products are summed across the
// LPK lanes with xor-shuffles; the chunk maximum across the warp's keys with
// two more. Each lane accumulates p*V for its own key into its own dims, so
// acc needs a cross-group reduction only once, at the end.
#pragma once

#include "common.cuh"

namespace pgqa {

template <int G> struct LanesPerKey {
    static constexpr int value = (G <= 4) ? 8 : 16;
};

template <int G> struct WarpAttn {
    static constexpr int LPK = LanesPerKey<G>::value;
    static constexpr int NSEG = kHeadDim / 8 / LPK; // 16-byte segments per lane and row
    static constexpr int DPL = NSEG * 8;            // dims per lane
    static constexpr int KPP = 32 / LPK;            // keys per pass
    static constexpr int PASSES = kChunkTokens / KPP;

    float q[G][DPL];   // query, times scale*log2(e)
    float acc[G][DPL]; // unnormalised sum of p*V over this lane group's keys
    float m[G];        // running max (base-2 units), identical in all lanes
    float l[G];        // sum of p over this lane group's keys

    __device__ __forceinline__ static int sub_lane() { return (threadIdx.x & 31) % LPK; }
    __device__ __forceinline__ static int group() { return (threadIdx.x & 31) / LPK; }
    // byte offset within a row of segment j owned by this lane
    __device__ __forceinline__ static int seg_byte(int j) { return (j * LPK + sub_lane()) * 16; }
    // head dimension of element e of segment j owned by this lane
    __device__ __forceinline__ static int seg_dim(int j) { return (j * LPK + sub_lane()) * 8; }

    // Load q rows [G][128] (bf16) and pre-scale; reset the state.
    __device__ __forceinline__ void init(const __nv_bfloat16 *q_rows, float scale_log2)
    {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int j = 0; j < NSEG; ++j) {
                const uint4 u = *reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const char *>(q_rows + h * kHeadDim) + seg_byte(j));
                float f[8];
                unpack8(u, f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q[h][j * 8 + e] = f[e] * scale_log2;
                    acc[h][j * 8 + e] = 0.f;
                }
            }
            m[h] = kEmptyMax;
            l[h] = 0.f;
        }
    }

    // Fold one chunk of up to 16 keys; rows >= n_valid are masked out (their
    // K and V are never used, whatever they hold). Rows are read through
    // `rows.key(row, byte)` / `rows.value(row, byte)`.
    template <class Rows> __device__ __forceinline__ void fold_chunk(const Rows &rows, int n_valid)
    {
        const int grp = group();
        float s[PASSES][G];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int row = ps * KPP + grp;
            float kf[DPL];
            if (!Rows::kGuard || row < n_valid) {
#pragma unroll
                for (int j = 0; j < NSEG; ++j)
                    unpack8(rows.key(row, seg_byte(j)), kf + 8 * j);
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e)
                    kf[e] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e)
                    d = fmaf(q[h][e], kf[e], d);
                s[ps][h] = d;
            }
        }
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int off = 1; off < LPK; off <<= 1)
                    s[ps][h] += __shfl_xor_sync(0xFFFFFFFFu, s[ps][h], off);
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps)
            if (ps * KPP + grp >= n_valid)
#pragma unroll
                for (int h = 0; h < G; ++h)
                    s[ps][h] = -INFINITY;

#pragma unroll
        for (int h = 0; h < G; ++h) {
            float cm = s[0][h];
#pragma unroll
            for (int ps = 1; ps < PASSES; ++ps)
                cm = fmaxf(cm, s[ps][h]);
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1)
                cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, off));
            const float mn = fmaxf(m[h], cm);
            if (mn > m[h]) { // warp-uniform: m and cm are the same in all lanes
                const float corr = exp2f(m[h] - mn);
                l[h] *= corr;
#pragma unroll
                for (int e = 0; e < DPL; ++e)
                    acc[h][e] *= corr;
                m[h] = mn;
            }
        }
        float p[PASSES][G];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                p[ps][h] = exp2f(s[ps][h] - m[h]); // masked: exp2(-inf) = 0
                l[h] += p[ps][h];
            }
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int row = ps * KPP + grp;
            if (row < n_valid) {
                float vf[DPL];
#pragma unroll
                for (int j = 0; j < NSEG; ++j)
                    unpack8(rows.value(row, seg_byte(j)), vf + 8 * j);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < DPL; ++e)
                        acc[h][e] = fmaf(p[ps][h], vf[e], acc[h][e]);
            }
        }
    }

    // Sum l and acc over the warp's lane groups; afterwards every lane holds
    // the warp's totals for its own dims.
    __device__ __forceinline__ void reduce_groups()
    {
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                l[h] += __shfl_xor_sync(0xFFFFFFFFu, l[h], off);
#pragma unroll
                for (int e = 0; e < DPL; ++e)
                    acc[h][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[h][e], off);
            }
        }
    }

    // Write this warp's state to a scratch record laid out
    // [G][kHeadDim] acc, then [G] m, then [G] l (floats). Call after
    // reduce_groups().
    __device__ __forceinline__ void store_record(float *rec) const
    {
        if (group() == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int j = 0; j < NSEG; ++j)
#pragma unroll
                    for (int e = 0; e < 8; e += 4)
                        *reinterpret_cast<float4 *>(rec + h * kHeadDim + seg_dim(j) + e) =
                            make_float4(acc[h][j * 8 + e], acc[h][j * 8 + e + 1],
                                        acc[h][j * 8 + e + 2], acc[h][j * 8 + e + 3]);
        }
        if ((threadIdx.x & 31) == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                rec[G * kHeadDim + h] = m[h];
                rec[G * kHeadDim + G + h] = l[h];
            }
        }
    }
};

// Floats in one warp-state record, padded to a multiple of 4 so that
// consecutive records stay 16-byte aligned for float4 stores.
template <int G> __host__ __device__ constexpr int record_floats()
{
    return G * kHeadDim + ((2 * G + 3) / 4) * 4;
}

// K/V rows of one chunk staged in shared memory: row r at base + r*256 bytes.
struct SmemRows {
    static constexpr bool kGuard = false; // rows past the valid count are staged but unused
    uint32_t k, v;
    __device__ __forceinline__ uint4 key(int row, int byte) const
    {
        return lds128(k + row * kRowBytes + byte);
    }
    __device__ __forceinline__ uint4 value(int row, int byte) const
    {
        return lds128(v + row * kRowBytes + byte);
    }
};

// K/V rows read straight from global memory with a row stride (bytes).
struct GlobalRows {
    static constexpr bool kGuard = true; // rows past the valid count may lie outside the buffer
    const char *k, *v;
    long stride;
    __device__ __forceinline__ uint4 key(int row, int byte) const
    {
        return ldg_stream128(k + row * stride + byte);
    }
    __device__ __forceinline__ uint4 value(int row, int byte) const
    {
        return ldg_stream128(v + row * stride + byte);
    }
};

} // namespace pgqa
