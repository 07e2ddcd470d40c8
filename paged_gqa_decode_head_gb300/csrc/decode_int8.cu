// decode_int8.cu -- paged GQA decode attention over an INT8 KV cache.
//
// "From Qwen3 math to CUDA kernels: a 0.6B inference runtime": s0.1 INT8
// values are multiplied by an FP32 scale and accumulated in FP32; s2.5/s2.6
// the attention itself; s10.1/s10.2 one CTA per (sequence, KV head,
// partition) serving all g query heads, partitions merged exactly (s9.1).
// The RTX 5090 residency page notes that on a bandwidth-bound path int8
// halves the bytes, which is what it buys here: a (position, KV head) costs
// 2 x 128 code bytes and two FP32 scales instead of 512 bytes.
//
// Cache: codes int8 [num_pages][Hkv][P][128] (symmetric, per row), scales
// float [num_pages][Hkv][P] for K and for V.
//
// GB300 design, as the bf16 kernel: one 288-thread CTA per SM, 9 warps each
// owning every 9th 16-position chunk and a ring of 3 stages; a chunk is two
// 2 KiB TMA tiles (K, V: 16 rows x 128 bytes, 128-byte swizzle) plus the
// chunk's 2 x 64 bytes of scales by bulk copy, all completing on one
// mbarrier. The fold runs fp16 tensor-core MMAs (m16n8k16) on codes
// converted in registers: ldmatrix hands a lane four consecutive bytes of a
// row, so the MMA's k index (S^T = K Q^T) and M index (O^T = V^T P^T) are
// taken in a fixed permutation of the 16 dims of a step -- the query is loaded
// in the same permutation and the output rows are stored back in dim order.
// Per-key K scales multiply the scores; per-key V scales are folded into P,
// which is split into fp16 hi + lo parts. Partition states go to the
// workspace and merge_kernel merges them.
#include <algorithm>
#include <cmath>
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace pgqa {
namespace {

__device__ unsigned g_flags_int8;

__device__ __forceinline__ void raise_flag8(unsigned f) { atomicOr(&g_flags_int8, f); }

constexpr int kWarps8 = 9;
constexpr int kStages8 = 6; // ring of stages per warp: two fold groups, one loading while the other folds
constexpr int kGroup8 = 3;  // chunks folded together
constexpr int kTile8 = kChunkTokens * 128;  // 16 rows x 128 int8 codes
constexpr int kStage8 = 2 * kTile8;         // K tile, V tile
constexpr int kScaleBytes8 = 2 * kChunkTokens * 4; // K scales, V scales
constexpr int kStageArea8 = kWarps8 * kStages8 * kStage8;
constexpr int kScaleOffset8 = kStageArea8;
constexpr int kBarOffset8 = kScaleOffset8 + kWarps8 * kStages8 * kScaleBytes8;
constexpr int kRowsOffset8 = kBarOffset8 + kWarps8 * kStages8 * 8;
constexpr int kSmem8 = 1024 /* alignment slack */ + kRowsOffset8 + kWarps8 * kStages8 * 4;

struct Int8Params {
    const uint16_t *q;
    const int32_t *block_table, *context_lens;
    const float *k_scale, *v_scale;
    float *out_f32;
    uint16_t *out_bf16;
    float *ws_m, *ws_l, *ws_acc;
    int Hq, Hkv, P, max_pages, num_pages, NP, ppp;
    float scale_log2;
};

// Per-warp online-softmax state on fp16 MMA fragments (transposed as in the
// bf16 kernel: the g <= 8 query heads are the N = 8 columns). Lane (g, t)
// holds heads 2t, 2t+1 for keys g and g+8 of a chunk; its O^T fragment rows
// are dims 16mt + 2g and 16mt + 2g + 1 (the permuted M index).
// With G <= 4 the lo parts of P ride in the spare N columns: column h < 4
// carries head h's hi part, column 4 + h its lo part (lanes t >= 2), so one
// PV MMA takes both; the two are added when the record is stored.
template <int G> struct Int8Warp {
    static constexpr bool kPackLo = G <= 4;
    uint32_t qb0[8], qb1[8]; // Q^T for k-step ks: dims 16ks+4t, +1 and 16ks+4t+2, +3 of head g (fp16x2)
    float o[8][4];
    float m[2], l[2];

    __device__ __forceinline__ void init(const uint16_t *q_rows)
    {
        const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (g < G) {
                const uint2 u = *reinterpret_cast<const uint2 *>(q_rows + g * kHeadDim + 16 * ks + 4 * t);
                qb0[ks] = pack_f16x2(bf16_lo(u.x), bf16_hi(u.x));
                qb1[ks] = pack_f16x2(bf16_lo(u.y), bf16_hi(u.y));
            } else {
                qb0[ks] = qb1[ks] = 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kEmptyMax;
        l[0] = l[1] = 0.f;
    }

    // Fold NC resident chunks: stage[c] is the shared address of chunk c's
    // K tile (its V tile follows), scl[c] its 32 scales (16 K, then 16 V),
    // rows[c] its valid rows.
    template <int NC>
    __device__ __forceinline__ void fold(const uint32_t (&stage)[kGroup8], const float *const (&scl)[kGroup8],
                                         const int (&rows)[kGroup8], float scale_log2)
    {
        const int lane = threadIdx.x & 31, g = lane >> 2;
        const int mq = lane >> 3, mr = lane & 7;
        // S^T = K Q^T: ldmatrix.x4 covers k-steps ks and ks+1 (units of 16
        // bytes): matrices (rows 0-7, unit ks), (rows 8-15, ks), (0-7, ks+1),
        // (8-15, ks+1); a lane receives bytes 4t..4t+3 of its row.
        float sa[NC][4], sb[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sa[c][e] = sb[c][e] = 0.f;
        const int krow = ((mq & 1) << 3) + mr;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            const int unit = 2 * kp + (mq >> 1);
            const uint32_t off = krow * 128 + ((unit ^ (krow & 7)) << 4);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t r[4];
                ldmatrix_x4(r, stage[c] + off);
#pragma unroll
                for (int h = 0; h < 2; ++h) { // k-step 2kp + h: matrices 2h (keys 0-7), 2h+1 (keys 8-15)
                    const uint32_t r0 = r[2 * h] ^ 0x80808080u, r1 = r[2 * h + 1] ^ 0x80808080u;
                    const uint32_t a[4] = {biased8x2_to_f16x2(r0, 0x100u), biased8x2_to_f16x2(r1, 0x100u),
                                           biased8x2_to_f16x2(r0, 0x302u), biased8x2_to_f16x2(r1, 0x302u)};
                    const int ks = 2 * kp + h;
                    mma_f16_16816(h ? sb[c] : sa[c], a, qb0[ks], qb1[ks]);
                }
            }
        }
        // scores: sc[c][e], e = 0 (key g, head 2t), 1 (key g, 2t+1), 2 (key g+8, 2t), 3 (key g+8, 2t+1)
        float sc[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float k0 = scl[c][g], k1 = scl[c][g + 8];
            sc[c][0] = (sa[c][0] + sb[c][0]) * k0 * scale_log2;
            sc[c][1] = (sa[c][1] + sb[c][1]) * k0 * scale_log2;
            sc[c][2] = (sa[c][2] + sb[c][2]) * k1 * scale_log2;
            sc[c][3] = (sa[c][3] + sb[c][3]) * k1 * scale_log2;
            if (g >= rows[c])
                sc[c][0] = sc[c][1] = -INFINITY;
            if (g + 8 >= rows[c])
                sc[c][2] = sc[c][3] = -INFINITY;
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
            float oc0 = c0, oc1 = c1;
            if constexpr (kPackLo) { // columns 4..7 belong to the heads of lane t - 2
                const float s0 = __shfl_xor_sync(0xFFFFFFFFu, c0, 2);
                const float s1 = __shfl_xor_sync(0xFFFFFFFFu, c1, 2);
                if (lane & 2) {
                    oc0 = s0;
                    oc1 = s1;
                }
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= oc0;
                o[mt][2] *= oc0;
                o[mt][1] *= oc1;
                o[mt][3] *= oc1;
            }
            m[0] = mn[0];
            m[1] = mn[1];
        }
        // P'^T = (p * v_scale of its key) as fp16 hi + lo, transposed into
        // the B operand layout; invalid keys contribute exactly 0 (their
        // scales may hold anything).
        uint32_t bh0[NC], bh1[NC], bl0[NC], bl1[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                p[e] = exp2f(sc[c][e] - m[e & 1]);
            l[0] += p[0] + p[2];
            l[1] += p[1] + p[3];
            const float v0 = g < rows[c] ? scl[c][16 + g] : 0.f;
            const float v1 = g + 8 < rows[c] ? scl[c][16 + g + 8] : 0.f;
            const float w0 = g < rows[c] ? p[0] * v0 : 0.f, w1 = g < rows[c] ? p[1] * v0 : 0.f;
            const float w2 = g + 8 < rows[c] ? p[2] * v1 : 0.f, w3 = g + 8 < rows[c] ? p[3] * v1 : 0.f;
            const uint32_t hi0 = pack_f16x2(w0, w1), hi1 = pack_f16x2(w2, w3);
            const uint32_t lo0 = pack_f16x2(w0 - f16_lo(hi0), w1 - f16_hi(hi0));
            const uint32_t lo1 = pack_f16x2(w2 - f16_lo(hi1), w3 - f16_hi(hi1));
            if constexpr (kPackLo) {
                const uint32_t lo0_src = __shfl_xor_sync(0xFFFFFFFFu, lo0, 2);
                const uint32_t lo1_src = __shfl_xor_sync(0xFFFFFFFFu, lo1, 2);
                bh0[c] = movmatrix_trans((lane & 2) ? lo0_src : hi0);
                bh1[c] = movmatrix_trans((lane & 2) ? lo1_src : hi1);
            } else {
                bh0[c] = movmatrix_trans(hi0);
                bh1[c] = movmatrix_trans(hi1);
                bl0[c] = movmatrix_trans(lo0);
                bl1[c] = movmatrix_trans(lo1);
            }
        }
        // O^T += V^T P'^T: ldmatrix.x4.trans covers units u and u+1 of the V
        // tile: matrices (keys 0-7, u), (keys 8-15, u), (0-7, u+1), (8-15, u+1).
        // A lane receives, for keys 2t, 2t+1, the bytes of dims 16u+2g and
        // 16u+2g+1: bytes {0, 2} are fragment row g, bytes {1, 3} row g + 8.
        const int vrow = ((mq & 1) << 3) + mr;
#pragma unroll
        for (int up = 0; up < 4; ++up) {
            const int unit = 2 * up + (mq >> 1);
            const uint32_t off = kTile8 + vrow * 128 + ((unit ^ (vrow & 7)) << 4);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t r[4];
                ldmatrix_x4_trans(r, stage[c] + off);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int mt = 2 * up + h;
                    const uint32_t r0 = r[2 * h] ^ 0x80808080u, r1 = r[2 * h + 1] ^ 0x80808080u;
                    const uint32_t a[4] = {biased8x2_to_f16x2(r0, 0x200u), biased8x2_to_f16x2(r0, 0x301u),
                                           biased8x2_to_f16x2(r1, 0x200u), biased8x2_to_f16x2(r1, 0x301u)};
                    mma_f16_16816(o[mt], a, bh0[c], bh1[c]);
                    if constexpr (!kPackLo)
                        mma_f16_16816(o[mt], a, bl0[c], bl1[c]);
                }
            }
        }
    }

    // Warp totals and record [G][128] O (dim order), [G] m, [G] l.
    __device__ __forceinline__ void store_record(float *rec)
    {
        const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
        if constexpr (kPackLo) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[mt][e] += __shfl_xor_sync(0xFFFFFFFFu, o[mt][e], 2);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 4);
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 8);
            l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 16);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = 2 * t + c;
            if (h < G) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    rec[h * kHeadDim + 16 * mt + 2 * g] = o[mt][c];
                    rec[h * kHeadDim + 16 * mt + 2 * g + 1] = o[mt][2 + c];
                }
                if (g == 0) {
                    rec[G * kHeadDim + h] = m[c];
                    rec[G * kHeadDim + G + h] = l[c];
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

template <int G>
__global__ void __launch_bounds__(kWarps8 * 32, 1)
    decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const Int8Params p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

    allow_dependent_launch();
    unsigned char *stages = smem + warp * kStages8 * kStage8;
    float *scales = reinterpret_cast<float *>(smem + kScaleOffset8) + warp * kStages8 * 2 * kChunkTokens;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOffset8) + warp * kStages8;
    int *stage_rows = reinterpret_cast<int *>(smem + kRowsOffset8) + warp * kStages8;
    if (lane == 0) {
        if (warp == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
#pragma unroll
        for (int s = 0; s < kStages8; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }

    const int part_tokens = p.ppp * p.P;
    const int tok0 = part * part_tokens;
    const int32_t *table = p.block_table + static_cast<size_t>(b) * p.max_pages;
    auto chunk_token = [&](int k) { return tok0 + (warp + k * kWarps8) * kChunkTokens; };
    int T = p.context_lens[b];
    if (T < 0 || T > p.max_pages * p.P) {
        if (part == 0 && threadIdx.x == 0)
            raise_flag8(PGQA_DEVERR_BAD_CONTEXT);
        T = 0;
    }
    const int n_parts = max(1, (T + part_tokens - 1) / part_tokens);
    if (part >= n_parts) {
        grid_dependency_wait();
        return;
    }
    const int tok1 = min(T, tok0 + part_tokens);
    const int n_chunks = max(0, (tok1 - tok0 + kChunkTokens - 1) / kChunkTokens);
    const int my_chunks = (n_chunks > warp) ? (n_chunks - 1 - warp) / kWarps8 + 1 : 0;
    __syncwarp();

    // the chunk holding position T-1 is written by the prologue this kernel
    // may overlap: it is requested after griddepcontrol.wait
    auto holds_new_token = [&](int k) { return chunk_token(k) + kChunkTokens > T - 1; };
    // Physical pages of this warp's chunks, 32 at a time: lane L caches the
    // entry of chunk 32*blk + L. Called by the whole (converged) warp.
    int tbl_blk = -1, tbl_val = -1;
    auto phys_of = [&](int k) {
        if ((k >> 5) != tbl_blk) {
            tbl_blk = k >> 5;
            const int kk = (tbl_blk << 5) + lane;
            tbl_val = kk < my_chunks ? table[chunk_token(kk) / p.P] : -1;
        }
        return __shfl_sync(0xFFFFFFFFu, tbl_val, k & 31);
    };
    auto issue = [&](int k, int phys, uint64_t policy) { // lane 0
        const int t = chunk_token(k);
        uint64_t *bar = &bars[k % kStages8];
        if (phys < 0 || phys >= p.num_pages) {
            raise_flag8(PGQA_DEVERR_BAD_PAGE);
            stage_rows[k % kStages8] = 0;
            mbar_arrive(bar);
            return;
        }
        stage_rows[k % kStages8] = min(kChunkTokens, tok1 - t);
        const int row = (phys * p.Hkv + kvh) * p.P + (t % p.P);
        unsigned char *dst = stages + (k % kStages8) * kStage8;
        float *sdst = scales + (k % kStages8) * 2 * kChunkTokens;
        mbar_arrive_expect_tx(bar, kStage8 + kScaleBytes8);
        tma_load_2d(dst, &tmap_k, 0, row, bar, policy);
        tma_load_2d(dst + kTile8, &tmap_v, 0, row, bar, policy);
        bulk_copy_g2s(sdst, p.k_scale + row, kChunkTokens * 4, bar, policy);
        bulk_copy_g2s(sdst + kChunkTokens, p.v_scale + row, kChunkTokens * 4, bar, policy);
    };

    const uint64_t policy = l2_evict_first_policy();
    const int first = min(kStages8, my_chunks);
    int first_phys[kStages8];
#pragma unroll
    for (int k = 0; k < kStages8; ++k)
        first_phys[k] = k < first ? phys_of(k) : -1;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages8; ++k)
            if (k < first && !holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    grid_dependency_wait();
    Int8Warp<G> st;
    st.init(p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * kHeadDim);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages8; ++k)
            if (k < first && holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    __syncwarp();

    bool ok = true;
    int k0 = 0;
    for (int nc; k0 < my_chunks; k0 += nc) {
        nc = min(kGroup8, my_chunks - k0);
        uint32_t stage_addr[kGroup8];
        const float *scl[kGroup8];
        int rows[kGroup8];
#pragma unroll
        for (int c = 0; c < kGroup8; ++c) {
            const int k = k0 + c;
            stage_addr[c] = smem_addr(stages + (k % kStages8) * kStage8);
            scl[c] = scales + (k % kStages8) * 2 * kChunkTokens;
            rows[c] = 0;
            if (c < nc) {
                const bool landed = mbar_wait_bounded(&bars[k % kStages8], (k / kStages8) & 1);
                if (!__all_sync(0xFFFFFFFFu, landed))
                    ok = false;
                rows[c] = stage_rows[k % kStages8];
            }
        }
        if (!ok)
            break;
        if (nc == 3)
            st.template fold<3>(stage_addr, scl, rows, p.scale_log2);
        else if (nc == 2)
            st.template fold<2>(stage_addr, scl, rows, p.scale_log2);
        else
            st.template fold<1>(stage_addr, scl, rows, p.scale_log2);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kGroup8; ++c) {
            const int k = k0 + c + kStages8;
            if (c < nc && k < my_chunks) {
                const int phys = phys_of(k);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue(k, phys, policy);
                }
            }
        }
        __syncwarp();
    }
    if (!ok) {
        if (lane == 0)
            raise_flag8(PGQA_DEVERR_WAIT_TIMEOUT);
        const int issued = min(my_chunks, k0 + kStages8);
        for (int kk = k0; kk < issued; ++kk)
            (void)mbar_wait_bounded(&bars[kk % kStages8], (kk / kStages8) & 1);
        st.clear();
    }
    __syncwarp();
    // every copy into this warp's stages has landed: they can hold its record
    st.store_record(reinterpret_cast<float *>(stages));
    __syncthreads();

    const size_t row0 = static_cast<size_t>(b) * p.Hq + kvh * G;
    for (int e = threadIdx.x; e < G * kHeadDim; e += kWarps8 * 32) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float M = kEmptyMax;
#pragma unroll
        for (int w = 0; w < kWarps8; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * kStages8 * kStage8);
            M = fmaxf(M, rec[G * kHeadDim + h]);
        }
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps8; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * kStages8 * kStage8);
            const float wt = exp2f(rec[G * kHeadDim + h] - M);
            L = fmaf(rec[G * kHeadDim + G + h], wt, L);
            O = fmaf(rec[h * kHeadDim + d], wt, O);
        }
        const size_t row = row0 + h;
        if (n_parts == 1) {
            const float o = L > 0.f ? O / L : 0.f;
            if (p.out_f32)
                p.out_f32[row * kHeadDim + d] = o;
            if (p.out_bf16)
                p.out_bf16[row * kHeadDim + d] = f32_to_bf16_bits(o);
        } else {
            const size_t idx = row * p.NP + part;
            if (d == 0) {
                p.ws_m[idx] = M; // base-2 units
                p.ws_l[idx] = L;
            }
            p.ws_acc[idx * kHeadDim + d] = O;
        }
    }
}

using EncodeTiledFn8 = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                    CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

EncodeTiledFn8 encode_fn8()
{
    static EncodeTiledFn8 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn8>(ptr);
    });
    return fn;
}

// An INT8 cache as a 2-D tensor [rows][128 bytes]; one box {128, 16} is a
// 16-row tile with 128-byte swizzle.
cudaError_t encode_int8_map(CUtensorMap *map, const void *base, long long rows)
{
    EncodeTiledFn8 fn = encode_fn8();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {128u, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {128u};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(kChunkTokens)};
    const cuuint32_t elem[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int G>
cudaError_t launch_int8_t(const CUtensorMap &mk, const CUtensorMap &mv, const Int8Params &kp, dim3 grid,
                          cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(decode_int8_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem8);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    return launch_pdl(decode_int8_kernel<G>, grid, dim3(kWarps8 * 32), kSmem8, stream, mk, mv, kp);
}

} // namespace

cudaError_t launch_decode_int8(const DecodeInt8Args &a, cudaStream_t stream)
{
    if (a.B == 0)
        return cudaSuccess;
    const int G = a.Hq / a.Hkv;
    CUtensorMap mk, mv;
    const long long rows = static_cast<long long>(a.num_pages) * a.Hkv * a.page_size;
    if (rows == 0)
        return cudaErrorInvalidValue;
    cudaError_t err = encode_int8_map(&mk, a.k_cache8, rows);
    if (err == cudaSuccess)
        err = encode_int8_map(&mv, a.v_cache8, rows);
    if (err != cudaSuccess)
        return err;
    Int8Params kp{};
    kp.q = a.q;
    kp.block_table = a.block_table;
    kp.context_lens = a.context_lens;
    kp.k_scale = a.k_scale;
    kp.v_scale = a.v_scale;
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
        const auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
        char *ws = reinterpret_cast<char *>(a.ws);
        kp.ws_m = reinterpret_cast<float *>(ws);
        kp.ws_l = reinterpret_cast<float *>(ws + a256(n * sizeof(float)));
        kp.ws_acc = reinterpret_cast<float *>(ws + 2 * a256(n * sizeof(float)));
    }
    const dim3 grid(a.num_partitions, a.Hkv, a.B);
    switch (G) {
    case 1: err = launch_int8_t<1>(mk, mv, kp, grid, stream); break;
    case 2: err = launch_int8_t<2>(mk, mv, kp, grid, stream); break;
    case 3: err = launch_int8_t<3>(mk, mv, kp, grid, stream); break;
    case 4: err = launch_int8_t<4>(mk, mv, kp, grid, stream); break;
    case 5: err = launch_int8_t<5>(mk, mv, kp, grid, stream); break;
    case 6: err = launch_int8_t<6>(mk, mv, kp, grid, stream); break;
    case 7: err = launch_int8_t<7>(mk, mv, kp, grid, stream); break;
    case 8: err = launch_int8_t<8>(mk, mv, kp, grid, stream); break;
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

size_t decode_int8_workspace_bytes(int B, int Hq, int num_partitions)
{
    if (num_partitions <= 1)
        return 0;
    const size_t n = static_cast<size_t>(B) * Hq * num_partitions;
    const auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    return 2 * a256(n * sizeof(float)) + a256(n * kHeadDim * sizeof(float));
}

cudaError_t read_flags_int8(unsigned *flags, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_flags_int8, sizeof(unsigned));
    if (err == cudaSuccess && clear) {
        const unsigned zero = 0;
        err = cudaMemcpyToSymbol(g_flags_int8, &zero, sizeof(unsigned));
    }
    return err;
}

} // namespace pgqa
