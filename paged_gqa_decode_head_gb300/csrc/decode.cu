// decode.cu -- paged GQA decode attention, split over KV partitions, and the
// exact partition merge.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime":
//   s10.1 one CTA per (sequence, KV head) serves all g query heads of the
//         group, so every K/V byte is read from HBM once;
//   s10.2 the history is cut into partitions, one CTA each, whose
//         (m_p, l_p, o_p) go to a preallocated fp32 scratch and are merged;
//   s9.1  the merge rescales every partition to the common maximum, which is
//         exact (not an approximation);
//   s12.1 / s12.2 multi-stage prefetch, aligned copies, masked tails,
//         swizzled shared memory against bank conflicts.
//
// GB300 design.
// * Grid = (partition, KV head, sequence), one 288-thread CTA per SM. Each of
//   the 9 warps owns every 9th 16-position chunk of the partition and a
//   private ring of 3 shared-memory stages (27 chunks = 216 KiB per CTA).
//   Grids of several waves with short partitions (a forced partition count)
//   run two CTAs per SM instead, 6 warps x 2 stages each, so that one CTA's
//   start and end overlap the other's streaming. Lane 0 of a warp issues
//   one 3-D TMA load per 4 KiB chunk of K and of V (16 rows, two 64-column
//   halves, 128-byte swizzle) that complete on the stage's mbarrier.
// * The warp folds its resident chunks together with tensor-core MMAs
//   (mma.sync m16n8k16, bf16 in, fp32 accumulate), transposed so the g <= 8
//   query heads fill the N = 8 columns: S^T = K Q^T, the online softmax on the
//   S^T fragments, then O^T += V^T P^T with P split into bf16 hi + lo parts
//   (~16 significant bits). ldmatrix reads the swizzled tiles without bank
//   conflicts; movmatrix turns P^T from the accumulator layout into the B
//   operand layout.
// * Programmatic dependent launch: a partition's first chunks are requested
//   before griddepcontrol.wait, so one layer's history streams in while the
//   previous kernels in the stream (the previous layer, this layer's prologue)
//   finish; the query and the chunk holding the new token are read after it.
//   With 27 chunks per SM a whole 8192-position, 8-head layer nearly fits;
//   such a latency-bound layer runs on nine tenths of the SMs (the rest take
//   the previous layer's merging CTAs) and its warps fold in pairs.
// * The warps' states are merged in shared memory; NP = 1 writes the output,
//   NP > 1 writes the partition state. With at most kFusedMergeMax
//   partitions the last CTA of each (sequence, KV head) to finish (a ticket
//   counter in the workspace, reset by that CTA) merges them; the others exit
//   at once, freeing their SM for the next layer. Larger NP use merge_kernel
//   (also launched with programmatic dependence).
#include <algorithm>
#include <cmath>
#include <mutex>

#include <cuda.h>
#include <type_traits>

#include "attn_core.cuh"
#include "head_norm_rope.cuh"
#include "launch.h"
#include "partition_merge.cuh"
#include "tensor_map.h"

namespace pgqa {
namespace {

__device__ unsigned g_flags_decode;

__device__ __forceinline__ void raise_flag(unsigned f) { atomicOr(&g_flags_decode, f); }

constexpr int kBoxBytes = kChunkTokens * 128;   // 16 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kStageBytes = 4 * kBoxBytes;      // K lo, K hi, V lo, V hi
constexpr int kFusedMergeMax = 64;              // partitions the last CTA merges itself

// CTA shape: kW warps, each with a ring of kS chunk stages, kCtas CTAs per
// SM. Shared memory (from a 1024-byte aligned base): the stages, one
// mbarrier and one valid-row count per stage, the partition ticket, the
// merge's mbarrier, the rotated query and the new K, V rows of the fused step.
template <int kW, int kS, int kCtas> struct Shape {
    static constexpr int kWarps = kW;
    static constexpr int kStages = kS;
    static constexpr int kCtasPerSm = kCtas;
    static constexpr int kThreads = kW * 32;
    static constexpr int kStageAreaBytes = kW * kS * kStageBytes;
    static constexpr int kBarOffset = kStageAreaBytes;
    static constexpr int kRowsOffset = kBarOffset + kW * kS * 8;
    static constexpr int kTicketOffset = (kRowsOffset + kW * kS * 4 + 7) & ~7;
    static constexpr int kMergeBarOffset = kTicketOffset + 8;
    static constexpr int kQBufOffset = (kMergeBarOffset + 8 + 15) & ~15;
    static constexpr int kPatchOffset = kQBufOffset + kMaxGroup * kHeadDim * 2;
    static constexpr int kSmem = 1024 /* alignment slack */ + kPatchOffset + 4 * kHeadDim;
    // The in-kernel merge copies the G x n partition accumulators of its
    // group into the stage area, followed by its scratch (weights, sums, a
    // float4 per thread); launch_decode falls back to merge_kernel when they
    // do not fit.
    static constexpr int kMergeScratchBytes = merge_scratch_bytes<kThreads, kFusedMergeMax>(kMaxGroup);
    static_assert(kSmem <= 232448, "at most 227 KB of shared memory per CTA");
    static_assert(kCtas * (kSmem + 1024) <= 233472, "228 KB of shared memory per SM, 1 KB reserved per CTA");
};
// One CTA per SM holding 27 staged chunks (216 KiB): across 152 SMs that is
// more than a whole 8192-position layer of one 8-head KV cache. Used for
// every grid that fits one wave and for long partitions.
using SoloShape = Shape<9, 3, 1>;
// Two CTAs per SM of 6 warps x 2 stages (96 KiB each): for grids of several
// waves with short partitions, where one CTA's start (table and context
// loads, first request) and end (merge, state write) overlap the other's
// streaming. B = 1, Hq = 32, T = 131072 with 512-position partitions (2048
// CTAs): 96.8 vs 113.3 us; 2048-position partitions 87.8 vs 95.0 us.
using PairShape = Shape<6, 2, 2>;
// Longest partition (positions) the two-CTA shape takes: B = 64 ragged
// contexts with 4096-position partitions run 1 % faster on SoloShape.
constexpr int kPairMaxPositions = 2048;

// Chunks per warp requested before the grid wait, measured on the 28-layer
// T = 8192 chain (NP = 15): the fused step does best with 2 (1: +0.7 us per
// layer, 3: +0.25 us), attention alone with all.
template <bool kFused, int kStages> constexpr int kPrewaitChunks = kFused && kStages > 2 ? 2 : kStages;

struct SplitParams {
    const uint16_t *q;
    const int32_t *block_table, *context_lens;
    float *out_f32;
    uint16_t *out_bf16;
    float *ws_m, *ws_l, *ws_acc;
    unsigned *tickets; // [B*Hkv] partition tickets (fused merge)
    int Hq, Hkv, P, max_pages, num_pages, NP, ppp;
    int G, M; // group size; new tokens per sequence (column n = query n / G, head n % G)
    int fused_merge;
    int walk; // decode_walk_kernel: partitions per CTA
    float scale_log2;
    // fused decode step only: the new token's raw heads and the prologue's
    // parameters; the kernel normalises/rotates q and appends K/V itself
    const uint16_t *q_raw, *k_new, *v_new, *gamma_q, *gamma_k;
    uint16_t *k_cache, *v_cache, *q_out;
    float eps;
    RopeFreqs freqs;
#ifdef PGQA_TIMELINE
    unsigned long long *tl; // timeline buffer, or NULL
    int tl_launch;          // this launch's index in it
#endif
};

// Row (of the [B][M][Hq] query / output arrays) of column n of KV head kvh;
// with one new token (kMulti = false) the columns are the heads kvh*G + n.
template <bool kMulti>
__device__ __forceinline__ size_t column_row(const SplitParams &p, int b, int kvh, int n)
{
    if constexpr (kMulti)
        return (static_cast<size_t>(b) * p.M + n / p.G) * p.Hq + kvh * p.G + n % p.G;
    else
        return static_cast<size_t>(b) * p.Hq + kvh * p.G + n;
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t *p)
{
    return *reinterpret_cast<const uint32_t *>(p);
}

// Per-warp online-softmax state on mma fragments, computed transposed so the
// g <= 8 query heads fill the mma's N = 8 columns instead of padding its M =
// 16 rows: S^T = K Q^T (A = 16 keys x 16 dims of K, B = Q^T) and
// O^T += V^T P^T (A = 16 dims x 16 keys of V^T, B = P^T). Lane (g, t) =
// (lane / 4, lane % 4) holds heads 2t and 2t+1 (valid when < G) for keys g
// and g+8 of a chunk, and O^T rows (dims) 16mt+g and 16mt+g+8.
//
// The NCOL <= 8 columns are (query, head) pairs: the g query heads of the KV
// head for the single-token step, and (query i, head h) at column i*g + h
// when M new tokens are decoded at once.
template <int NCOL> struct MmaWarp {
    uint32_t qb0[8], qb1[8]; // B = Q^T: column g, dims 16ks+2t..+1 and 16ks+8+2t..+1 (bf16x2)
    float o[8][4];           // O^T m-tile mt: [dim 16mt+g][2t], [..][2t+1], [dim 16mt+g+8][2t], [..][2t+1]
    float m[2];              // running max of columns 2t, 2t+1 (base-2 units)
    float l[2];              // sum of p of columns 2t, 2t+1 over this lane's keys

    // q_row: the query row of this lane's column g (lane / 4), or NULL when
    // g >= NCOL.
    __device__ __forceinline__ void init(const uint16_t *q_row)
    {
        const int lane = threadIdx.x & 31, t = lane & 3;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qb0[ks] = q_row ? ld_u32(q_row + 16 * ks + 2 * t) : 0u;
            qb1[ks] = q_row ? ld_u32(q_row + 16 * ks + 8 + 2 * t) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kEmptyMax;
        l[0] = l[1] = 0.f;
    }

    // Fold NC resident chunks at once (their MMAs and loads interleave):
    // stage[c] is the shared address of chunk c's four swizzled boxes; keys
    // from row lim0[c] (lim1[c]) on are masked out for column 2t (2t+1) --
    // the chunk's valid rows, cut further by a column's causal limit.
    template <int NC, bool kPerColumn, int N>
    __device__ __forceinline__ void fold(const uint32_t (&stage)[N], const int (&lim0)[N], const int (&lim1)[N],
                                         float scale_log2)
    {
        static_assert(NC <= N, "one stage per folded chunk");
        const int lane = threadIdx.x & 31, g = lane >> 2;
        const int mq = lane >> 3, mr = lane & 7; // ldmatrix: matrix index, row within it

        // S^T = K Q^T over 8 k-steps of 16 dims, two accumulators per chunk
        // (even and odd k-steps) to shorten the dependent MMA chains.
        float sa[NC][4], sb[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sa[c][e] = sb[c][e] = 0.f;
        const int k_key = ((mq & 1) << 3) + mr;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int unit = (2 * ks + (mq >> 1)) & 7;
            const uint32_t off = (ks >> 2) * kBoxBytes + k_key * 128 + ((unit ^ mr) << 4);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t a[4];
                ldmatrix_x4(a, stage[c] + off);
                mma_bf16_16816((ks & 1) ? sb[c] : sa[c], a, qb0[ks], qb1[ks]);
            }
        }
        // sc[c][e]: e = 0 (key g, column 2t), 1 (key g, 2t+1), 2 (key g+8, 2t), 3 (key g+8, 2t+1)
        float sc[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[c][e] = (sa[c][e] + sb[c][e]) * scale_log2;
            if constexpr (kPerColumn) {
                if (g >= lim0[c])
                    sc[c][0] = -INFINITY;
                if (g >= lim1[c])
                    sc[c][1] = -INFINITY;
                if (g + 8 >= lim0[c])
                    sc[c][2] = -INFINITY;
                if (g + 8 >= lim1[c])
                    sc[c][3] = -INFINITY;
            } else { // every column has the chunk's valid rows, lim0
                if (g >= lim0[c])
                    sc[c][0] = sc[c][1] = -INFINITY;
                if (g + 8 >= lim0[c])
                    sc[c][2] = sc[c][3] = -INFINITY;
            }
        }
        float mn[2];
        bool grow = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float cm = fmaxf(sc[0][h], sc[0][2 + h]);
#pragma unroll
            for (int c = 1; c < NC; ++c)
                cm = fmaxf(cm, fmaxf(sc[c][h], sc[c][2 + h]));
            cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 4));
            cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 8));
            cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 16));
            mn[h] = fmaxf(m[h], cm);
            grow |= mn[h] > m[h];
        }
        if (__any_sync(0xFFFFFFFFu, grow)) {
            const float c0 = exp2f(m[0] - mn[0]), c1 = exp2f(m[1] - mn[1]);
            l[0] *= c0;
            l[1] *= c1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= c0;
                o[mt][2] *= c0;
                o[mt][1] *= c1;
                o[mt][3] *= c1;
            }
            m[0] = mn[0];
            m[1] = mn[1];
        }
        // P^T as bf16 hi + lo (hi carries 8 significant bits, lo the next 8),
        // transposed from the accumulator layout into the B operand layout.
        uint32_t bh0[NC], bh1[NC], bl0[NC], bl1[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                p[e] = exp2f(sc[c][e] - m[e & 1]); // masked: exp2(-inf) = 0
            l[0] += p[0] + p[2];
            l[1] += p[1] + p[3];
            const uint32_t hi0 = pack_bf16x2(p[0], p[1]), hi1 = pack_bf16x2(p[2], p[3]);
            const uint32_t lo0 = pack_bf16x2(p[0] - bf16_lo(hi0), p[1] - bf16_hi(hi0));
            const uint32_t lo1 = pack_bf16x2(p[2] - bf16_lo(hi1), p[3] - bf16_hi(hi1));
            bh0[c] = movmatrix_trans(hi0);
            bh1[c] = movmatrix_trans(hi1);
            bl0[c] = movmatrix_trans(lo0);
            bl1[c] = movmatrix_trans(lo1);
        }
        const int v_key = ((mq >> 1) << 3) + mr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int dtile = 2 * mt + (mq & 1); // 8-dim block this lane addresses
            const uint32_t off =
                2 * kBoxBytes + (dtile >> 3) * kBoxBytes + v_key * 128 + (((dtile & 7) ^ mr) << 4);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t a[4];
                ldmatrix_x4_trans(a, stage[c] + off);
                mma_bf16_16816(o[mt], a, bh0[c], bh1[c]);
                mma_bf16_16816(o[mt], a, bl0[c], bl1[c]);
            }
        }
    }

    // Warp totals: reduce l over the 8 lanes sharing t; write the record
    // [NCOL][128] O, then [NCOL] m, then [NCOL] l.
    __device__ __forceinline__ void store_record(float *rec)
    {
        const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 4);
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 8);
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 16);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = 2 * t + c;
            if (h < NCOL) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    rec[h * kHeadDim + 16 * mt + g] = o[mt][c];
                    rec[h * kHeadDim + 16 * mt + g + 8] = o[mt][2 + c];
                }
                if (g == 0) {
                    rec[NCOL * kHeadDim + h] = m[c];
                    rec[NCOL * kHeadDim + NCOL + h] = l[c];
                }
            }
        }
    }

    __device__ __forceinline__ void clear()
    {
        m[0] = m[1] = kEmptyMax;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
};

// With more (column, dim) elements than threads, each column's maximum,
// weights and sum are formed once (one thread per column) instead of for every
// element, with the same operations in the same order (M = 4 fused step, 8
// columns: 11.04 -> 10.91 us per layer), and a thread folds four dims.
template <int NCOL, int kWarps> constexpr bool kSharesWeights = NCOL * kHeadDim > kWarps * 32;

// Folds the kWarps records of one partition -- warp w's at rec0 + w *
// rec_stride bytes: [NCOL][128] O, then [NCOL] m, then [NCOL] l -- into the
// partition's (m, l, acc) state, or into the outputs when it is the
// sequence's only partition, with weights 2^(m_w - M) against the largest M.
// wts holds [NCOL][kWarps] weights, then M [NCOL], L [NCOL] when the weights
// are shared. Called by all kWarps * 32 threads of the CTA once every record
// is visible to all of them.
template <int NCOL, int kWarps, bool kMulti>
__device__ __forceinline__ void fold_records(const SplitParams &p, const unsigned char *rec0, int rec_stride,
                                             float *wts, int b, int kvh, int part, int n_parts)
{
    constexpr bool kSharedWeights = kSharesWeights<NCOL, kWarps>;
    if constexpr (kSharedWeights) {
        if (threadIdx.x < NCOL) {
            const int h = threadIdx.x;
            float M = kEmptyMax;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float *rec = reinterpret_cast<const float *>(rec0 + w * rec_stride);
                M = fmaxf(M, rec[NCOL * kHeadDim + h]);
            }
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float *rec = reinterpret_cast<const float *>(rec0 + w * rec_stride);
                const float wt = exp2f(rec[NCOL * kHeadDim + h] - M);
                L = fmaf(rec[NCOL * kHeadDim + NCOL + h], wt, L);
                wts[h * kWarps + w] = wt;
            }
            wts[NCOL * kWarps + h] = M;
            wts[NCOL * kWarps + NCOL + h] = L;
        }
        __syncthreads();
    }
    // The CTA's state of column h, dims d .. d + cnt - 1: the outputs when it
    // is the sequence's only partition, else its partition state.
    const auto put_state = [&](int h, int d, float M, float L, const float *O, auto cnt) {
        constexpr int kCnt = decltype(cnt)::value;
        const size_t row = column_row<kMulti>(p, b, kvh, h);
        if (n_parts == 1) {
            float o[kCnt];
#pragma unroll
            for (int i = 0; i < kCnt; ++i)
                o[i] = L > 0.f ? O[i] / L : 0.f;
            if constexpr (kCnt == 4) {
                if (p.out_f32)
                    *reinterpret_cast<float4 *>(p.out_f32 + row * kHeadDim + d) = make_float4(o[0], o[1], o[2], o[3]);
                if (p.out_bf16)
                    *reinterpret_cast<uint2 *>(p.out_bf16 + row * kHeadDim + d) =
                        make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
            } else {
                if (p.out_f32)
                    p.out_f32[row * kHeadDim + d] = o[0];
                if (p.out_bf16)
                    p.out_bf16[row * kHeadDim + d] = f32_to_bf16_bits(o[0]);
            }
        } else {
            const size_t idx = row * p.NP + part;
            if (d == 0) {
                p.ws_m[idx] = M; // base-2 units (private workspace format)
                p.ws_l[idx] = L;
            }
            if constexpr (kCnt == 4)
                *reinterpret_cast<float4 *>(p.ws_acc + idx * kHeadDim + d) = make_float4(O[0], O[1], O[2], O[3]);
            else
                p.ws_acc[idx * kHeadDim + d] = O[0];
        }
    };
    if constexpr (kSharedWeights) {
        // four consecutive dims per thread
        for (int e = threadIdx.x; e < NCOL * (kHeadDim / 4); e += kWarps * 32) {
            const int h = e / (kHeadDim / 4);
            const int d = 4 * (e % (kHeadDim / 4));
            float O[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float4 r =
                    *reinterpret_cast<const float4 *>(rec0 + w * rec_stride + (h * kHeadDim + d) * 4);
                const float wt = wts[h * kWarps + w];
                O[0] = fmaf(r.x, wt, O[0]);
                O[1] = fmaf(r.y, wt, O[1]);
                O[2] = fmaf(r.z, wt, O[2]);
                O[3] = fmaf(r.w, wt, O[3]);
            }
            put_state(h, d, wts[NCOL * kWarps + h], wts[NCOL * kWarps + NCOL + h], O,
                      std::integral_constant<int, 4>{});
        }
    } else {
        for (int e = threadIdx.x; e < NCOL * kHeadDim; e += kWarps * 32) {
            const int h = e / kHeadDim;
            const int d = e % kHeadDim;
            float M = kEmptyMax, L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float *rec = reinterpret_cast<const float *>(rec0 + w * rec_stride);
                M = fmaxf(M, rec[NCOL * kHeadDim + h]);
            }
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float *rec = reinterpret_cast<const float *>(rec0 + w * rec_stride);
                const float wt = exp2f(rec[NCOL * kHeadDim + h] - M);
                L = fmaf(rec[NCOL * kHeadDim + NCOL + h], wt, L);
                O = fmaf(rec[h * kHeadDim + d], wt, O);
            }
            put_state(h, d, M, L, &O, std::integral_constant<int, 1>{});
        }
    }
}

// The last CTA of a (sequence, KV head) to finish merges the n (2..64)
// partition states of its columns (partition_merge.cuh).
template <int NCOL, bool kMulti, int kThreads>
__device__ __forceinline__ void merge_in_last_cta(const SplitParams &p, int b, int kvh, int n,
                                                  unsigned char *smem, uint64_t *bar)
{
    const auto row_of = [&](int c) { return column_row<kMulti>(p, b, kvh, c); };
    if (!merge_partitions_in_cta<NCOL, kThreads, kFusedMergeMax>(p.ws_m, p.ws_l, p.ws_acc, p.NP, n, row_of,
                                                                     p.out_f32, p.out_bf16, smem, bar) &&
        threadIdx.x == 0)
        raise_flag(PGQA_DEVERR_WAIT_TIMEOUT); // the merge's copy never landed: outputs left alone
}

// kFused = true: the whole decode step of one layer (qk_norm_rope_append
// then decode attention) in one launch. Each CTA normalises and rotates the
// query heads it serves; the warp whose chunk holds position T-1 computes the
// new K row, appends K and V to the cache and patches the row into its staged
// chunk, so every history chunk can be requested before griddepcontrol.wait.
// NCOL = M * G columns; kMulti: M > 1 new tokens (not fused), each column
// with its own causal limit.
template <int NCOL, bool kFused, bool kMulti, typename S>
__global__ void __launch_bounds__(S::kThreads, S::kCtasPerSm)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const SplitParams p)
{
    constexpr int kWarps = S::kWarps, kStages = S::kStages;
    constexpr int kBarOffset = S::kBarOffset, kRowsOffset = S::kRowsOffset, kTicketOffset = S::kTicketOffset;
    constexpr int kMergeBarOffset = S::kMergeBarOffset, kQBufOffset = S::kQBufOffset;
    constexpr int kPatchOffset = S::kPatchOffset;
    constexpr int kPrewait = kPrewaitChunks<kFused, kStages>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;

    allow_dependent_launch();
    TL_STAMP(0);
    unsigned char *stages = smem + warp * kStages * kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOffset) + warp * kStages;
    if (lane == 0) {
        if (warp == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }

    const int part_tokens = p.ppp * p.P;
    const int tok0 = part * part_tokens;
    const int32_t *table = p.block_table + static_cast<size_t>(b) * p.max_pages;
    auto chunk_token = [&](int k) { return tok0 + (warp + k * kWarps) * kChunkTokens; };
    // The first 32 table entries of this warp's chunks are loaded before the
    // context length is known (any entry below max_pages may be read), so the
    // two loads overlap.
    int tbl_blk = 0;
    int tbl_val;
    {
        const int page = chunk_token(lane) / p.P;
        tbl_val = (chunk_token(lane) < tok0 + part_tokens && page < p.max_pages) ? table[page] : -1;
    }
    int T = p.context_lens[b];
    // M new tokens sit at positions T - M .. T - 1 (M = 1: the decode step)
    if (T < (kFused || p.M > 1 ? p.M : 0) || T > p.max_pages * p.P) {
        if (part == 0 && threadIdx.x == 0)
            raise_flag(PGQA_DEVERR_BAD_CONTEXT);
        T = 0;
    }
    const int n_parts = max(1, (T + part_tokens - 1) / part_tokens);
    if (part >= n_parts) {
        grid_dependency_wait(); // keep the chain ordered even when idle
        return;
    }
    const int tok1 = min(T, tok0 + part_tokens);
    const int n_chunks = max(0, (tok1 - tok0 + kChunkTokens - 1) / kChunkTokens);
    const int my_chunks = (n_chunks > warp) ? (n_chunks - 1 - warp) / kWarps + 1 : 0;

    int *stage_rows = reinterpret_cast<int *>(smem + kRowsOffset) + warp * kStages;
    __syncwarp();

    // Chunks holding the new positions T - M .. T - 1 are written by the
    // prologue this kernel may overlap, so they are requested only after
    // griddepcontrol.wait (the fused step patches its row into shared memory
    // itself instead).
    auto holds_new_token = [&](int k) {
        return (!kFused || kMulti) && chunk_token(k) + kChunkTokens > T - p.M;
    };
    // Physical pages of this warp's chunks, 32 at a time: lane L caches the
    // entry of chunk 32*blk + L. Called by the whole (converged) warp.
    auto phys_of = [&](int k) {
        if ((k >> 5) != tbl_blk) {
            tbl_blk = k >> 5;
            const int kk = (tbl_blk << 5) + lane;
            tbl_val = kk < my_chunks ? table[chunk_token(kk) / p.P] : -1;
        }
        return __shfl_sync(0xFFFFFFFFu, tbl_val, k & 31);
    };
    // Lane 0 requests chunk k (phys from phys_of) and records its valid rows.
    auto issue = [&](int k, int phys, uint64_t policy) {
        const int t = chunk_token(k);
        uint64_t *bar = &bars[k % kStages];
        if (phys < 0 || phys >= p.num_pages) {
            raise_flag(PGQA_DEVERR_BAD_PAGE);
            stage_rows[k % kStages] = 0;
            mbar_arrive(bar); // complete the phase with no data; the keys are masked
            return;
        }
        stage_rows[k % kStages] = min(kChunkTokens, tok1 - t);
        const int row = (phys * p.Hkv + kvh) * p.P + (t % p.P);
        unsigned char *dst = stages + (k % kStages) * kStageBytes;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_3d(dst, &tmap_k, 0, row, 0, bar, policy);
        tma_load_3d(dst + 2 * kBoxBytes, &tmap_v, 0, row, 0, bar, policy);
    };

    const uint64_t policy = l2_evict_first_policy();
    const int first = min(kStages, my_chunks);
    int first_phys[kStages];
#pragma unroll
    for (int k = 0; k < kStages; ++k)
        first_phys[k] = k < first ? phys_of(k) : -1;
    TL_STAMP(1);
    // Only the first kPrewait chunks of each warp are requested before
    // griddepcontrol.wait: in the fused step the rest would queue in the
    // memory system ahead of the previous layer's merge and this layer's
    // query loads, which sit on the critical path of the layer chain.
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages; ++k)
            if (k < first && k < kPrewait && !holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    TL_STAMP(2);

    // fused step: what the prologue needs that no earlier kernel writes
    // (gains, rotation, the append slot) is prepared before the wait.
    // Single token (kMulti = false): warps < G rotate the query heads; once
    // every warp has its query, the warp owning the chunk of position T-1
    // computes the new K row, appends K and V and keeps the row in shared
    // memory to patch it into its staged chunk. M tokens (kMulti):
    // warp w < NCOL rotates column w (token w / G, head w % G) and warp w < M
    // appends token w at T - M + w; chunks holding new positions are
    // requested only once every append is done.
    const bool has_q = kFused && T > 0 && warp < NCOL;
    const int q_pos = kMulti ? T - p.M + warp / p.G : T - 1; // position of column `warp`
    const bool has_tok = kFused && kMulti && T > 0 && warp < p.M;
    const int tok_pos = T - p.M + warp; // kMulti: position of token `warp`
    const int pos = T - 1;              // single token
    int new_chunk = -1; // single token: index k of the chunk holding pos in this warp's sequence, or -1
    int new_phys = -1;
    if (kFused && !kMulti && T > 0 && pos >= tok0 && pos < tok1) {
        const int c_idx = (pos - tok0) / kChunkTokens;
        if (c_idx % kWarps == warp) {
            new_chunk = c_idx / kWarps;
            new_phys = table[pos / p.P];
        }
    }
    if (has_tok) {
        // token `warp`: its slot, appended by every partition's CTA that owns
        // it -- the CTA whose range holds tok_pos
        if (tok_pos >= tok0 && tok_pos < tok1)
            new_phys = table[tok_pos / p.P];
    }
    const bool appends = kMulti ? (has_tok && tok_pos >= tok0 && tok_pos < tok1) : new_chunk >= 0;
    HeadRope rope, rope_k;
    float gain_q[4], gain_k[4];
    if (has_q)
        rope.init(q_pos, p.freqs);
    if (appends) {
        if constexpr (kMulti)
            rope_k.init(tok_pos, p.freqs);
        else
            rope_k = has_q ? rope : (rope.init(pos, p.freqs), rope);
    }
    if (has_q)
        load_head(p.gamma_q, gain_q);
    if (appends)
        load_head(p.gamma_k, gain_k);

    grid_dependency_wait();
    TL_STAMP(3);

    // The new tokens' q, k, v come from the previous kernels: load them now,
    // ahead of the remaining bulk requests.
    const size_t qrow = has_q ? column_row<kMulti>(p, b, kvh, warp) * kHeadDim : 0;
    const size_t krow = ((static_cast<size_t>(b) * (kMulti ? p.M : 1) + (kMulti ? warp : 0)) * p.Hkv + kvh) * kHeadDim;
    float xq[4], xk[4];
    uint16_t new_v[4] = {0, 0, 0, 0};
    MmaWarp<NCOL> st;
    const int col = lane >> 2; // this lane's B-operand column
    if (has_q)
        load_head(p.q_raw + qrow, xq);
    if (appends) {
        load_head(p.k_new + krow, xk);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            new_v[i] = p.v_new[krow + lane + 32 * i];
    }
    if constexpr (!kFused)
        st.init(col < NCOL ? p.q + column_row<kMulti>(p, b, kvh, col) * kHeadDim : nullptr);
    // the fused multi-token step requests new-token chunks after the appends
    constexpr bool kDeferNew = kFused && kMulti;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages; ++k)
            if (k < first && (k >= kPrewait || holds_new_token(k)) &&
                !(kDeferNew && holds_new_token(k)))
                issue(k, first_phys[k], policy);
    }
    __syncwarp();

    // fused step: normalise and rotate q and the new K rows, append K and V.
    if constexpr (kFused) {
        uint16_t *q_buf = reinterpret_cast<uint16_t *>(smem + kQBufOffset);
        if (has_q) {
            norm_rope_apply(xq, gain_q, p.eps, rope);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint16_t bits = f32_to_bf16_bits(xq[i]);
                q_buf[warp * kHeadDim + lane + 32 * i] = bits;
                if (part == 0 && p.q_out)
                    p.q_out[qrow + lane + 32 * i] = bits;
            }
        }
        if (kMulti && appends) {
            // M tokens: appended before the barrier, their chunks requested after it
            norm_rope_apply(xk, gain_k, p.eps, rope_k);
            if (new_phys >= 0 && new_phys < p.num_pages) {
                const size_t slot =
                    ((static_cast<size_t>(new_phys) * p.Hkv + kvh) * p.P + tok_pos % p.P) * kHeadDim;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p.k_cache[slot + lane + 32 * i] = f32_to_bf16_bits(xk[i]);
                    p.v_cache[slot + lane + 32 * i] = new_v[i];
                }
            } else if (lane == 0) {
                raise_flag(PGQA_DEVERR_BAD_PAGE);
            }
            if constexpr (kDeferNew)
                fence_proxy_async_global(); // the appends before the bulk reads of their chunks
        }
        __syncthreads();
        if constexpr (kDeferNew) {
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kStages; ++k)
                    if (k < first && holds_new_token(k))
                        issue(k, first_phys[k], policy);
            }
            __syncwarp();
        }
        st.init(col < NCOL ? q_buf + col * kHeadDim : nullptr);
        TL_STAMP(4);
        if (!kMulti && appends) {
            // single token: off the other warps' path; the row waits in
            // shared memory for the patch of its staged chunk
            uint16_t *patch = reinterpret_cast<uint16_t *>(smem + kPatchOffset);
            norm_rope_apply(xk, gain_k, p.eps, rope_k);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                patch[lane + 32 * i] = f32_to_bf16_bits(xk[i]);
                patch[kHeadDim + lane + 32 * i] = new_v[i];
            }
            if (new_phys >= 0 && new_phys < p.num_pages) {
                const size_t slot = ((static_cast<size_t>(new_phys) * p.Hkv + kvh) * p.P + pos % p.P) * kHeadDim;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p.k_cache[slot + lane + 32 * i] = patch[lane + 32 * i];
                    p.v_cache[slot + lane + 32 * i] = new_v[i];
                }
            } else if (lane == 0) {
                raise_flag(PGQA_DEVERR_BAD_PAGE);
            }
            __syncwarp();
        }
    }

    // Causal limit (exclusive position) of this lane's columns 2t and 2t+1:
    // query i sees positions up to T - M + i.
    int qlim0 = T, qlim1 = T;
    if constexpr (kMulti) {
        const int c_lo = 2 * (lane & 3);
        if (c_lo < NCOL)
            qlim0 = T - p.M + 1 + c_lo / p.G;
        if (c_lo + 1 < NCOL)
            qlim1 = T - p.M + 1 + (c_lo + 1) / p.G;
    }

    // Chunks are consumed in groups (one stage per chunk); the group's stages
    // are refilled together once it has been folded. A warp with few chunks
    // (the latency-bound layer chain) folds pairs: the first pair (its early
    // requests) is folded while the third chunk is in flight and its stages
    // are refilled sooner (8.74 vs 9.06 us per layer for the fused step); one
    // with many folds whole rings. The grouping depends only on the chunk
    // count, so equal inputs give equal bits.
    const int group = my_chunks <= 2 * kStages ? 2 : kStages;
    bool ok = true;
    int k0 = 0;
    for (int nc; k0 < my_chunks; k0 += nc) {
        nc = min(group, my_chunks - k0);
        uint32_t stage_addr[kStages];
        int rows[kStages], lim0[kStages], lim1[kStages];
#pragma unroll
        for (int c = 0; c < kStages; ++c) {
            const int k = k0 + c;
            stage_addr[c] = smem_addr(stages + (k % kStages) * kStageBytes);
            rows[c] = lim0[c] = lim1[c] = 0;
            if (c < nc) {
                const bool landed = mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1);
                if (!__all_sync(0xFFFFFFFFu, landed))
                    ok = false;
                if (k == 1)
                    TL_STAMP(5);
                if (k == my_chunks - 1)
                    TL_STAMP_LATEST(6);
                rows[c] = stage_rows[k % kStages];
                if (kFused && k == new_chunk && rows[c] > 0) {
                    // the staged copy predates the append: put the new row in
                    // (word w < 128 of the patch: K dims 2w, 2w+1 for w < 64,
                    // then V dims 2(w-64), 2(w-64)+1)
                    const int r = (T - 1) % kChunkTokens;
                    unsigned char *stage = stages + (k % kStages) * kStageBytes;
                    const uint32_t *patch = reinterpret_cast<const uint32_t *>(smem + kPatchOffset);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int w = lane + 32 * i;
                        const int d = 2 * (w & 63);
                        const int x = d & 63, u = x >> 3;
                        const int off = (w >> 6) * 2 * kBoxBytes + (d >> 6) * kBoxBytes + r * 128 +
                                        ((u ^ (r & 7)) << 4) + (x & 7) * 2;
                        *reinterpret_cast<uint32_t *>(stage + off) = patch[w];
                    }
                    __syncwarp();
                }
                lim0[c] = rows[c];
                lim1[c] = rows[c];
                if constexpr (kMulti) {
                    lim0[c] = min(rows[c], qlim0 - chunk_token(k));
                    lim1[c] = min(rows[c], qlim1 - chunk_token(k));
                }
                if (rows[c] < kChunkTokens) {
                    // Rows past the history (all rows of a chunk whose page
                    // was refused) may hold anything, even NaN: zero their V
                    // so that p = 0 times V stays 0 in the MMA.
                    unsigned char *stage = stages + (k % kStages) * kStageBytes;
                    const int n_units = (kChunkTokens - rows[c]) * 16;
                    for (int u = lane; u < n_units; u += 32) {
                        const int row = rows[c] + u / 16;
                        const int box = 2 + ((u >> 3) & 1);
                        *reinterpret_cast<uint4 *>(stage + box * kBoxBytes + row * 128 + (u & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok)
            break;
        if constexpr (kStages >= 3) {
            if (nc == 3)
                st.template fold<3, kMulti>(stage_addr, lim0, lim1, p.scale_log2);
            else if (nc == 2)
                st.template fold<2, kMulti>(stage_addr, lim0, lim1, p.scale_log2);
            else
                st.template fold<1, kMulti>(stage_addr, lim0, lim1, p.scale_log2);
        } else {
            if (nc == 2)
                st.template fold<2, kMulti>(stage_addr, lim0, lim1, p.scale_log2);
            else
                st.template fold<1, kMulti>(stage_addr, lim0, lim1, p.scale_log2);
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kStages; ++c) {
            const int k = k0 + c + kStages;
            if (c < nc && k < my_chunks) {
                const int phys = phys_of(k);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue(k, phys, policy);
                }
            }
        }
    }
    if (!ok) {
        // A copy never completed: flag it, wait (bounded) for the copies
        // still in flight into this warp's stages, and contribute nothing.
        if (lane == 0)
            raise_flag(PGQA_DEVERR_WAIT_TIMEOUT);
        const int issued = min(my_chunks, k0 + kStages);
        for (int kk = k0; kk < issued; ++kk)
            (void)mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1);
        st.clear();
    }

    __syncwarp();
    // Every copy into this warp's stages has landed: they can hold its record.
    st.store_record(reinterpret_cast<float *>(stages));
    __syncthreads();
    TL_STAMP(7);

    constexpr int kWeightsOffset = 8192; // in warp 0's stages, past its record
    static_assert(!kSharesWeights<NCOL, kWarps> || (NCOL * kHeadDim + 2 * NCOL) * 4 <= kWeightsOffset,
                  "record overlaps weights");
    static_assert(!kSharesWeights<NCOL, kWarps> ||
                      kWeightsOffset + (NCOL * kWarps + 2 * NCOL) * 4 <= kStages * kStageBytes,
                  "weights past warp 0's stages");
    fold_records<NCOL, kWarps, kMulti>(p, smem, kStages * kStageBytes, reinterpret_cast<float *>(smem + kWeightsOffset),
                                       b, kvh, part, n_parts);
    if (n_parts == 1 || !p.fused_merge)
        return;

    TL_STAMP(8);
    // Ticket: the CTA that finishes last for this (sequence, KV head) merges.
    // The barrier orders every thread's partial-state stores before thread
    // 0's release; its acquire (when last) orders the other CTAs' stores
    // before the merge's loads, which the second barrier extends to all
    // threads.
    unsigned *ticket_slot = reinterpret_cast<unsigned *>(smem + kTicketOffset);
    __syncthreads();
    unsigned *ticket = p.tickets + static_cast<size_t>(b) * p.Hkv + kvh;
    if (threadIdx.x == 0)
        *ticket_slot = atomic_add_acq_rel_gpu(ticket, 1u);
    __syncthreads();
    TL_STAMP(9);
    if (*ticket_slot != static_cast<unsigned>(n_parts - 1))
        return;
    merge_in_last_cta<NCOL, kMulti, S::kThreads>(p, b, kvh, n_parts, smem,
                                                 reinterpret_cast<uint64_t *>(smem + kMergeBarOffset));
#ifdef PGQA_TIMELINE
    __syncthreads();
    TL_STAMP(10);
#endif
    if (threadIdx.x == 0)
        *ticket = 0u; // ready for the next call
}

// Attention alone over many short partitions (more CTAs than one wave of the
// two-CTA shape, partition states merged by merge_kernel), walked: each CTA
// takes a run of consecutive partitions of one (sequence, KV head), and its
// warps keep requesting the next partition's chunks while they finish the
// current one, so no CTA start (table, context, first requests) or end
// (records, state write) leaves an SM without bytes in flight. Within a
// partition the chunks, their warps (chunk c of the partition: warp
// c % kWarps), the fold pairs and the record fold are the two-CTA shape's,
// so every partition state, and the merged outputs, equal that kernel's bit
// for bit; decode_step_paged keeps the two-CTA shape for such grids and still
// matches the two launches.
// Shared memory: the stages, their mbarriers and valid-row counts, the
// warps' records of the current partition, the record fold's weights and a
// flag that a copy never landed.
template <int NCOL, int kS, int kCtas> struct WalkShape {
    static constexpr int kWarps = PairShape::kWarps;
    static constexpr int kStages = kS;
    static constexpr int kCtasPerSm = kCtas;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kBarOffset = kWarps * kStages * kStageBytes;
    static constexpr int kRowsOffset = kBarOffset + kWarps * kStages * 8;
    static constexpr int kRecFloats = (NCOL * kHeadDim + 2 * NCOL + 3) & ~3;
    static constexpr int kRecOffset = (kRowsOffset + kWarps * kStages * 4 + 15) & ~15;
    static constexpr int kWtsOffset = kRecOffset + kWarps * kRecFloats * 4;
    static constexpr int kAbortedOffset = kWtsOffset + (NCOL * kWarps + 2 * NCOL) * 4;
    static constexpr int kSmem = 1024 /* alignment slack */ + kAbortedOffset + 16;
    static_assert(kSmem <= 232448, "at most 227 KB of shared memory per CTA");
    static_assert(kCtas * (kSmem + 1024) <= 233472, "228 KB of shared memory per SM, 1 KB reserved per CTA");
};
// Two CTAs per SM of 6 warps x 2 stages and their records (NCOL <= 4: for
// g = 5, 6 the records leave no room for two, and one CTA per SM streams
// less than the two-CTA shape, which those grids keep).
constexpr int kWalkMaxCols = 4;
template <int NCOL> using WalkShapeFor = WalkShape<NCOL, 2, 2>;

template <int NCOL, typename S>
__global__ void __launch_bounds__(S::kThreads, S::kCtasPerSm)
    decode_walk_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const SplitParams p)
{
    constexpr int kWarps = S::kWarps, kStages = S::kStages, kRec = S::kRecFloats;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;

    allow_dependent_launch();
    unsigned char *stages = smem + warp * kStages * kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBarOffset) + warp * kStages;
    int *stage_rows = reinterpret_cast<int *>(smem + S::kRowsOffset) + warp * kStages;
    float *recs = reinterpret_cast<float *>(smem + S::kRecOffset); // [kWarps][kRec]
    volatile int *aborted = reinterpret_cast<volatile int *>(smem + S::kAbortedOffset);
    if (lane == 0) {
        if (warp == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }

    const int part_tokens = p.ppp * p.P; // a multiple of the 16-position chunk (P >= 16)
    const int cpp = part_tokens / kChunkTokens;
    const int32_t *table = p.block_table + static_cast<size_t>(b) * p.max_pages;
    int T = p.context_lens[b];
    if (T < 0 || T > p.max_pages * p.P) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            raise_flag(PGQA_DEVERR_BAD_CONTEXT);
        T = 0;
    }
    const int n_parts = max(1, (T + part_tokens - 1) / part_tokens);
    const int j0 = blockIdx.x * p.walk;
    const int j1 = min(n_parts, j0 + p.walk);
    if (threadIdx.x == 0)
        *aborted = 0;
    __syncthreads();
    if (j0 >= j1) {
        grid_dependency_wait(); // keep the chain ordered even when idle
        return;
    }

    // This warp's chunks, partition after partition: nkf in each full
    // partition of the run, nk_last in a last, shorter one (the sequence's
    // end); chunk r of the walk is chunk k of partition j, position
    // j * part_tokens + (warp + k * kWarps) * 16.
    const auto owned = [&](int cnt) { return cnt > warp ? (cnt - 1 - warp) / kWarps + 1 : 0; };
    const int n_full = max(0, min(j1, T / part_tokens) - j0);
    const bool has_last = j1 - j0 > n_full;
    const int nkf = owned(cpp);
    const int nk_last = has_last ? owned((T - (j1 - 1) * part_tokens + kChunkTokens - 1) / kChunkTokens) : 0;
    const int total = nkf * n_full + nk_last;
    const auto chunk_pos = [&](int r) {
        const int in_full = nkf * n_full;
        const int j = r < in_full ? j0 + r / nkf : j0 + n_full;
        const int k = r < in_full ? r % nkf : r - in_full;
        return j * part_tokens + (warp + k * kWarps) * kChunkTokens;
    };
    // Physical pages of this warp's chunks, 32 at a time: lane L caches the
    // entry of chunk 32*blk + L. Called by the whole (converged) warp.
    int tbl_blk = -1, tbl_val = -1;
    const auto phys_of = [&](int r) {
        if ((r >> 5) != tbl_blk) {
            tbl_blk = r >> 5;
            const int rr = (tbl_blk << 5) + lane;
            tbl_val = rr < total ? table[chunk_pos(rr) / p.P] : -1;
        }
        return __shfl_sync(0xFFFFFFFFu, tbl_val, r & 31);
    };
    // Lane 0 requests chunk r (phys from phys_of) and records its valid rows
    // (partitions are whole chunks: only the sequence's end cuts one short).
    const auto issue = [&](int r, int phys, uint64_t policy) {
        const int t = chunk_pos(r);
        uint64_t *bar = &bars[r % kStages];
        if (phys < 0 || phys >= p.num_pages) {
            raise_flag(PGQA_DEVERR_BAD_PAGE);
            stage_rows[r % kStages] = 0;
            mbar_arrive(bar); // complete the phase with no data; the keys are masked
            return;
        }
        stage_rows[r % kStages] = min(kChunkTokens, T - t);
        const int row = (phys * p.Hkv + kvh) * p.P + (t % p.P);
        unsigned char *dst = stages + (r % kStages) * kStageBytes;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_3d(dst, &tmap_k, 0, row, 0, bar, policy);
        tma_load_3d(dst + 2 * kBoxBytes, &tmap_v, 0, row, 0, bar, policy);
    };
    // The chunk holding the new position T-1 is written by the prologue this
    // kernel may overlap: it is requested after griddepcontrol.wait.
    const auto holds_new_token = [&](int r) { return chunk_pos(r) + kChunkTokens > T - 1; };

    const uint64_t policy = l2_evict_first_policy();
    const int first = min(kStages, total);
    int first_phys[kStages];
#pragma unroll
    for (int k = 0; k < kStages; ++k)
        first_phys[k] = k < first ? phys_of(k) : -1;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages; ++k)
            if (k < first && !holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    grid_dependency_wait();
    MmaWarp<NCOL> st;
    const int col = lane >> 2; // this lane's B-operand column
    st.init(col < NCOL ? p.q + column_row<false>(p, b, kvh, col) * kHeadDim : nullptr);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages; ++k)
            if (k < first && holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    __syncwarp();

    bool ok = true;
    int r = 0; // next chunk of the walk to fold
    int issued = first;
    for (int j = j0; j < j1; ++j) {
        const int nk = j - j0 < n_full ? nkf : nk_last;
        // the partition's chunks in pairs, as the two-CTA shape folds them
        for (int k0 = 0, nc; ok && k0 < nk; k0 += nc) {
            nc = min(2, nk - k0);
            uint32_t stage_addr[2];
            int lim[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int rr = r + c;
                stage_addr[c] = smem_addr(stages + (rr % kStages) * kStageBytes);
                lim[c] = 0;
                if (c < nc) {
                    const bool landed = mbar_wait_bounded(&bars[rr % kStages], (rr / kStages) & 1);
                    if (!__all_sync(0xFFFFFFFFu, landed))
                        ok = false;
                    lim[c] = stage_rows[rr % kStages];
                    if (lim[c] < kChunkTokens) {
                        // rows past the history may hold anything, even NaN:
                        // zero their V so that p = 0 times V stays 0
                        unsigned char *stage = stages + (rr % kStages) * kStageBytes;
                        const int n_units = (kChunkTokens - lim[c]) * 16;
                        for (int u = lane; u < n_units; u += 32) {
                            const int row = lim[c] + u / 16;
                            const int box = 2 + ((u >> 3) & 1);
                            *reinterpret_cast<uint4 *>(stage + box * kBoxBytes + row * 128 + (u & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        __syncwarp();
                    }
                }
            }
            if (!ok)
                break;
            if (nc == 2)
                st.template fold<2, false>(stage_addr, lim, lim, p.scale_log2);
            else
                st.template fold<1, false>(stage_addr, lim, lim, p.scale_log2);
            __syncwarp();
            // the folded stages take the walk's next chunks, whatever their partition
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int rn = r + c + kStages;
                if (c < nc && rn < total) {
                    const int phys = phys_of(rn);
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        issue(rn, phys, policy);
                    }
                    issued = rn + 1;
                }
            }
            r += nc;
        }
        if (!ok && lane == 0)
            *aborted = 1;
        // The partition's records, folded as the two-CTA shape folds them;
        // every warp's next chunks are in flight meanwhile.
        st.store_record(recs + warp * kRec);
        st.clear();
        __syncthreads();
        if (*aborted)
            break; // every thread sees the same flag after the barrier
        fold_records<NCOL, kWarps, false>(p, reinterpret_cast<const unsigned char *>(recs), kRec * 4,
                                          reinterpret_cast<float *>(smem + S::kWtsOffset), b, kvh, j, n_parts);
        __syncthreads();
    }
    if (*aborted) {
        // A copy never landed: flag it and wait (bounded) for the copies
        // still in flight into this warp's stages.
        if (lane == 0)
            raise_flag(PGQA_DEVERR_WAIT_TIMEOUT);
        for (int rr = r; rr < issued; ++rr)
            (void)mbar_wait_bounded(&bars[rr % kStages], (rr / kStages) & 1);
    }
}

struct MergeParams {
    const float *m, *l, *acc;
    int Hq, NP;
    int M; // query rows per sequence are M * Hq (M new tokens)
    float *out_f32;
    uint16_t *out_bf16;
    const int32_t *context_lens;
    int P, ppp, max_pages;
};

constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeRound = 16; // partitions per warp whose loads are in flight together

// One CTA per (sequence, query head). Warp w folds partitions w, w+16, ...,
// kMergeRound at a time: all loads of a round are issued before any is used,
// and the round is folded into the warp's running (M, L, O) like the online
// softmax update (lane i owns dims 4i..4i+3); up to 256 partitions take one
// round trip to memory. The 16 warps' states are then merged through shared
// memory.
template <bool kBase2>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p)
{
    __shared__ float red_m[kMergeWarps];
    __shared__ float red_l[kMergeWarps];
    __shared__ float4 red_o[kMergeWarps][32];
    const int row = blockIdx.x; // b * Hq + h
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    allow_dependent_launch();
    grid_dependency_wait();
    int np = p.NP;
    if (p.context_lens) {
        const int b = row / (p.M * p.Hq);
        int T = p.context_lens[b];
        // the split kernel's test of a bad context (M new tokens need T >= M)
        if (T < (p.M > 1 ? p.M : 0) || T > p.max_pages * p.P)
            T = 0;
        const int part_tokens = p.ppp * p.P;
        np = min(np, max(1, (T + part_tokens - 1) / part_tokens));
        if (np == 1)
            return; // a single partition wrote this sequence's output itself
    }
    const float *m = p.m + static_cast<size_t>(row) * p.NP;
    const float *l = p.l + static_cast<size_t>(row) * p.NP;
    const float4 *acc = reinterpret_cast<const float4 *>(p.acc + static_cast<size_t>(row) * p.NP * kHeadDim);
    const float to_base2 = kBase2 ? 1.f : kLog2e;

    float M = kEmptyMax, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = warp; i0 < np; i0 += kMergeWarps * kMergeRound) {
        float mi[kMergeRound], li[kMergeRound];
        float4 ai[kMergeRound];
#pragma unroll
        for (int r = 0; r < kMergeRound; ++r) {
            const int i = i0 + r * kMergeWarps;
            const bool in = i < np;
            mi[r] = in ? __ldcg(m + i) * to_base2 : kEmptyMax;
            li[r] = in ? __ldcg(l + i) : 0.f;
            ai[r] = in ? __ldcg(acc + static_cast<size_t>(i) * (kHeadDim / 4) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mn = M;
#pragma unroll
        for (int r = 0; r < kMergeRound; ++r)
            mn = fmaxf(mn, mi[r]);
        const float corr = exp2f(M - mn);
        L *= corr;
        O.x *= corr, O.y *= corr, O.z *= corr, O.w *= corr;
#pragma unroll
        for (int r = 0; r < kMergeRound; ++r) {
            const float wt = exp2f(mi[r] - mn);
            L = fmaf(li[r], wt, L);
            O.x = fmaf(ai[r].x, wt, O.x);
            O.y = fmaf(ai[r].y, wt, O.y);
            O.z = fmaf(ai[r].z, wt, O.z);
            O.w = fmaf(ai[r].w, wt, O.w);
        }
        M = mn;
    }
    red_o[warp][lane] = O;
    if (lane == 0) {
        red_m[warp] = M;
        red_l[warp] = L;
    }
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
        const int d = threadIdx.x;
        float Mt = red_m[0];
#pragma unroll
        for (int w = 1; w < kMergeWarps; ++w)
            Mt = fmaxf(Mt, red_m[w]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            const float wt = exp2f(red_m[w] - Mt);
            Ls = fmaf(red_l[w], wt, Ls);
            Os = fmaf(reinterpret_cast<const float *>(&red_o[w][0])[d], wt, Os);
        }
        const float out = Ls > 0.f ? Os / Ls : 0.f;
        if (p.out_f32)
            p.out_f32[static_cast<size_t>(row) * kHeadDim + d] = out;
        if (p.out_bf16)
            p.out_bf16[static_cast<size_t>(row) * kHeadDim + d] = f32_to_bf16_bits(out);
    }
}

constexpr int kMaxDevices = 64;

// A paged cache seen as a 3-D tensor [2 halves][num_pages * Hkv * P rows]
// [64 bf16]: element (x, row, half) is column 64*half + x of that row. One
// box {64, 16, 2} is a whole 16-row chunk, landing in shared memory as the
// 16 rows of columns 0-63 followed by the 16 rows of columns 64-127, each
// 128-byte line swizzled (128-byte swizzle), so ldmatrix reads it without
// bank conflicts; one TMA instruction moves a 4 KiB chunk of K (or V).
cudaError_t encode_cache_map(CUtensorMap *map, const void *base, long long rows)
{
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), 2u};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes), 128u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(kChunkTokens), 2u};
    const cuuint32_t elem[3] = {1u, 1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NCOL, bool kFused, bool kMulti, typename S>
cudaError_t launch_split_t(const CUtensorMap &mk, const CUtensorMap &mv, const SplitParams &kp,
                           dim3 grid, cudaStream_t stream)
{
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= kMaxDevices || !configured[dev]) {
        err = cudaFuncSetAttribute(decode_mma_kernel<NCOL, kFused, kMulti, S>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
        if (err != cudaSuccess)
            return err;
        if (dev < kMaxDevices)
            configured[dev] = true;
    }
    return launch_pdl(decode_mma_kernel<NCOL, kFused, kMulti, S>, grid, dim3(S::kThreads), S::kSmem, stream,
                      mk, mv, kp);
}

// pair: the two-CTA shape (single token, NCOL <= its warps; the caller checks).
template <int NCOL>
cudaError_t launch_split(const CUtensorMap &mk, const CUtensorMap &mv, const SplitParams &kp,
                         dim3 grid, bool fused, bool pair, cudaStream_t stream)
{
    if (kp.M > 1)
        return fused ? launch_split_t<NCOL, true, true, SoloShape>(mk, mv, kp, grid, stream)
                     : launch_split_t<NCOL, false, true, SoloShape>(mk, mv, kp, grid, stream);
    if constexpr (NCOL <= PairShape::kWarps) {
        if (pair)
            return fused ? launch_split_t<NCOL, true, false, PairShape>(mk, mv, kp, grid, stream)
                         : launch_split_t<NCOL, false, false, PairShape>(mk, mv, kp, grid, stream);
    }
    return fused ? launch_split_t<NCOL, true, false, SoloShape>(mk, mv, kp, grid, stream)
                 : launch_split_t<NCOL, false, false, SoloShape>(mk, mv, kp, grid, stream);
}

template <int NCOL>
cudaError_t launch_walk(const CUtensorMap &mk, const CUtensorMap &mv, const SplitParams &kp, dim3 grid,
                        cudaStream_t stream)
{
    using S = WalkShapeFor<NCOL>;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= kMaxDevices || !configured[dev]) {
        err = cudaFuncSetAttribute(decode_walk_kernel<NCOL, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
        if (err != cudaSuccess)
            return err;
        if (dev < kMaxDevices)
            configured[dev] = true;
    }
    return launch_pdl(decode_walk_kernel<NCOL, S>, grid, dim3(S::kThreads), S::kSmem, stream, mk, mv, kp);
}

// Partitions per CTA of the walked grid, or 0 when walking does not apply:
// attention alone over a grid the two-CTA shape would run in several waves,
// merged by merge_kernel, with g <= 4 and few enough (sequence, KV head)
// pairs that runs of partitions fill at least 7/8 of the walked shape's CTA
// slots (two per SM).
int walk_partitions(bool pair, bool fused_merge, bool fused, int NCOL, int B, int Hkv, int num_partitions,
                    int sm_count)
{
    if (!pair || fused_merge || fused || NCOL > kWalkMaxCols)
        return 0;
    const long heads = static_cast<long>(B) * Hkv;
    const long slots = static_cast<long>(sm_count > 0 ? sm_count : 1) * WalkShapeFor<1>::kCtasPerSm;
    if (heads > slots)
        return 0;
    const long per_head = slots / heads;
    if (per_head * heads * 8 < slots * 7)
        return 0;
    const int walk = static_cast<int>((num_partitions + per_head - 1) / per_head);
    return walk >= 2 ? walk : 0;
}

// The two-CTA shape takes single-token grids of more than one wave (of one
// CTA per SM) whose partitions are short; the fused step and attention alone
// follow the same rule, so they keep giving equal bits.
bool use_pair_shape(int NCOL, int M, int B, int Hkv, int num_partitions, int part_positions, int sm_count)
{
    return M == 1 && NCOL <= PairShape::kWarps && num_partitions > 1 && part_positions <= kPairMaxPositions &&
           static_cast<long>(B) * Hkv * num_partitions > static_cast<long>(sm_count > 0 ? sm_count : 1);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

} // namespace

int choose_partitions(int B, int Hkv, int page_size, int max_pages, int requested, int sm_count)
{
    if (max_pages <= 0)
        return 1;
    long np;
    if (requested > 0) {
        np = requested;
    } else {
        // Pick NP minimising waves x (positions per CTA + a per-CTA cost):
        // with (b, KV head) units = B * Hkv and one CTA per SM, a wave runs
        // `slots` CTAs, each streaming ceil(max_pages / NP) pages; starting a
        // CTA (table and context loads, the first request's latency) costs
        // about as much as streaming kCtaCostPositions positions. Partitions
        // stay at least 128 positions long so the merge is amortised, and at
        // most ~4096 positions when the units alone fill a wave (the model
        // counts every sequence at max_pages, which overstates the work of a
        // ragged batch and would pick too few partitions).
        // The cost constant fits NP sweeps on GB300: B = 1 at T = 131072
        // wants one full wave (NP = 19), B = 2 NP = 8 or 9, B = 4 NP = 4,
        // B = 16 NP = 1, and B = 64 ragged contexts up to 32768 any NP from 4
        // to 12 (NP = 2: 4 % slower).
        constexpr long kCtaCostPositions = 600;
        const long units = static_cast<long>(B) * Hkv;
        const long slots = static_cast<long>(sm_count > 0 ? sm_count : 1) * SoloShape::kCtasPerSm;
        const long lo = std::max(1, 128 / page_size);
        const long max_np = std::max<long>(1, std::min<long>((max_pages + lo - 1) / lo, 2 * slots));
        const long hi_pages = std::max(1, 4096 / page_size);
        const long min_np = units >= slots ? std::min(max_np, (max_pages + hi_pages - 1) / hi_pages) : 1;
        long best = 0;
        double best_cost = 0.0;
        for (long n = min_np; n <= max_np; ++n) {
            const long ppp = (max_pages + n - 1) / n;
            if (n > min_np && (max_pages + ppp - 1) / ppp != n)
                continue; // the same split as a smaller n
            const long waves = (units * n + slots - 1) / slots;
            const double cost = static_cast<double>(waves) * (ppp * page_size + kCtaCostPositions);
            if (best == 0 || cost < best_cost) {
                best = n;
                best_cost = cost;
            }
        }
        // A layer that fits one wave with each partition inside one CTA's
        // ring (the T = 8192 layer chain) is bound by its chain of latencies,
        // not by bandwidth: there, leave a tenth of the SMs free for the CTAs
        // that merge (which hold their SM while the next layer starts) and
        // merge fewer partitions. B = 1, T = 8192 on GB300: NP = 17 instead of
        // 19 is 16 % faster for the bf16 fused step, 8 % for attention alone
        // and 15 % for the INT8 fused step; at T = 32768 and 131072, or B = 2,
        // a full wave stays best.
        const long best_ppp = (max_pages + best - 1) / best;
        if (units * best <= slots &&
            best_ppp * page_size <= SoloShape::kWarps * SoloShape::kStages * kChunkTokens)
            best = std::min(best, std::max<long>(1, slots * 9 / 10 / units));
        np = best;
    }
    np = std::min<long>(std::max<long>(np, 1), std::min(max_pages, kMaxPartitions));
    const long ppp = (max_pages + np - 1) / np;
    return static_cast<int>((max_pages + ppp - 1) / ppp);
}

EncodeTiledFn tensor_map_encoder()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

size_t decode_ticket_bytes(int B, int Hkv)
{
    return align256(static_cast<size_t>(B) * Hkv * sizeof(unsigned));
}

// Workspace (NP > 1): partition tickets [B*Hkv] (zero before first use;
// every completed call leaves them zero), then m, l [B*Hq*NP] and acc
// [B*Hq*NP*128] (fp32, no initial value needed); with M new tokens per
// sequence pass M * Hq as Hq.
size_t decode_workspace_bytes(int B, int Hkv, int Hq, int num_partitions)
{
    if (num_partitions <= 1)
        return 0;
    const size_t n = static_cast<size_t>(B) * Hq * num_partitions;
    return decode_ticket_bytes(B, Hkv) + 2 * align256(n * sizeof(float)) +
           align256(n * kHeadDim * sizeof(float));
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream)
{
    const int G = a.Hq / a.Hkv;
    const int M = a.M > 0 ? a.M : 1;
    const int NCOL = G * M; // (query, head) columns of one KV head, <= 8 (checked by the caller)
    CUtensorMap mk, mv;
    const long long rows = static_cast<long long>(a.num_pages) * a.Hkv * a.page_size;
    if (rows == 0)
        return cudaErrorInvalidValue;
    cudaError_t err = encode_cache_map(&mk, a.k_cache, rows);
    if (err == cudaSuccess)
        err = encode_cache_map(&mv, a.v_cache, rows);
    if (err != cudaSuccess)
        return err;
    SplitParams kp{};
    kp.q = a.q;
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
#ifdef PGQA_TIMELINE
    kp.tl = timeline_buffer();
    kp.tl_launch = timeline_next_launch();
#endif
    const bool pair = use_pair_shape(NCOL, M, a.B, a.Hkv, a.num_partitions, a.pages_per_part * a.page_size,
                                     a.sm_count);
    const long merge_bytes = static_cast<long>(NCOL) * a.num_partitions * kHeadDim * 4 +
                             (pair ? PairShape::kMergeScratchBytes : SoloShape::kMergeScratchBytes);
    kp.fused_merge =
        a.num_partitions <= kFusedMergeMax &&
                merge_bytes <= (pair ? PairShape::kStageAreaBytes : SoloShape::kStageAreaBytes)
            ? 1
            : 0;
    if (a.fused) {
        kp.q_raw = a.q_raw;
        kp.k_new = a.k_new;
        kp.v_new = a.v_new;
        kp.gamma_q = a.gamma_q;
        kp.gamma_k = a.gamma_k;
        kp.k_cache = const_cast<uint16_t *>(a.k_cache);
        kp.v_cache = const_cast<uint16_t *>(a.v_cache);
        kp.q_out = a.q_out;
        kp.eps = a.eps;
        kp.freqs = make_rope_freqs(a.rope_theta);
    }
    if (a.num_partitions > 1) {
        const size_t n = static_cast<size_t>(a.B) * M * a.Hq * a.num_partitions;
        char *ws = reinterpret_cast<char *>(a.ws);
        kp.tickets = reinterpret_cast<unsigned *>(ws);
        ws += decode_ticket_bytes(a.B, a.Hkv);
        kp.ws_m = reinterpret_cast<float *>(ws);
        kp.ws_l = reinterpret_cast<float *>(ws + align256(n * sizeof(float)));
        kp.ws_acc = reinterpret_cast<float *>(ws + 2 * align256(n * sizeof(float)));
    }
    dim3 grid(a.num_partitions, a.Hkv, a.B);
    kp.G = G;
    kp.M = M;
    kp.walk = walk_partitions(pair, kp.fused_merge != 0, a.fused, NCOL, a.B, a.Hkv, a.num_partitions, a.sm_count);
    if (kp.walk) {
        grid.x = (a.num_partitions + kp.walk - 1) / kp.walk;
        switch (NCOL) { // <= kWalkMaxCols
        case 1: err = launch_walk<1>(mk, mv, kp, grid, stream); break;
        case 2: err = launch_walk<2>(mk, mv, kp, grid, stream); break;
        case 3: err = launch_walk<3>(mk, mv, kp, grid, stream); break;
        case 4: err = launch_walk<4>(mk, mv, kp, grid, stream); break;
        default: return cudaErrorInvalidValue;
        }
    } else {
    switch (NCOL) {
    case 1: err = launch_split<1>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 2: err = launch_split<2>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 3: err = launch_split<3>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 4: err = launch_split<4>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 5: err = launch_split<5>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 6: err = launch_split<6>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 7: err = launch_split<7>(mk, mv, kp, grid, a.fused, pair, stream); break;
    case 8: err = launch_split<8>(mk, mv, kp, grid, a.fused, pair, stream); break;
    default: return cudaErrorInvalidValue;
    }
    }
    if (err != cudaSuccess || a.num_partitions <= 1 || kp.fused_merge)
        return err;
    MergeArgs ma{};
    ma.m = kp.ws_m;
    ma.l = kp.ws_l;
    ma.acc = kp.ws_acc;
    ma.B = a.B;
    ma.Hq = a.Hq;
    ma.NP = a.num_partitions;
    ma.M = M;
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
    mp.M = a.M > 0 ? a.M : 1;
    mp.out_f32 = a.out_f32;
    mp.out_bf16 = reinterpret_cast<uint16_t *>(a.out_bf16);
    mp.context_lens = a.context_lens;
    mp.P = a.page_size;
    mp.ppp = a.pages_per_part;
    mp.max_pages = a.max_pages;
    const unsigned rows = static_cast<unsigned>(a.B) * mp.M * a.Hq;
    if (a.context_lens)
        return launch_pdl(merge_kernel<true>, dim3(rows), dim3(kMergeThreads), 0, stream, mp);
    return launch_pdl(merge_kernel<false>, dim3(rows), dim3(kMergeThreads), 0, stream, mp);
}

namespace {

// One thread waits on an mbarrier that nothing completes: the bounded wait
// gives up after kWaitLimitNs and raises the same flag as a copy that never
// lands, so the failure path can be exercised without a fault.
__global__ void wait_selftest_kernel()
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0)
        return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0))
        raise_flag(PGQA_DEVERR_WAIT_TIMEOUT);
}

} // namespace

cudaError_t launch_wait_selftest(cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

#ifdef PGQA_TIMELINE
unsigned long long *g_timeline_buf = nullptr; // the attached buffer
int g_timeline_launches = 1, g_timeline_next = 0;

unsigned long long *timeline_buffer() { return g_timeline_buf; }

int timeline_next_launch()
{
    const int i = g_timeline_next;
    g_timeline_next = (g_timeline_next + 1) % g_timeline_launches;
    return i;
}

// Attach (or, with NULL, detach) the timeline buffer: `launches` slots of
// [CTAs][kTimelineSlots] u64, filled in turn by the following split-kernel
// launches of either kernel (captured graphs keep the slot they were
// captured with).
extern "C" int pgqa_timeline_attach(unsigned long long *buf, int launches)
{
    g_timeline_buf = buf;
    g_timeline_launches = launches > 0 ? launches : 1;
    g_timeline_next = 0;
    return kTimelineSlots;
}
#endif

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
