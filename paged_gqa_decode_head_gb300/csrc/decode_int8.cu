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
// GB300 design, as the bf16 kernel: one CTA per SM whose warps each own every
// kW-th 16-position chunk of the partition and a private ring of stages (12
// warps x 3 stages for short partitions, 16 warps x 3 for long ones, and
// four or two CTAs per SM of 4 or 8 warps x 3 for grids of several waves:
// see Shape8); a chunk is two 2 KiB TMA tiles (K, V:
// 16 rows x 128 bytes, 128-byte swizzle) plus the chunk's 2 x 64 bytes of
// scales, all completing on one mbarrier (one TMA load for both tiles and
// one for both scale rows when the caller's buffers allow it). The fold runs fp16 tensor-core MMAs (m16n8k16) on codes
// converted in registers: ldmatrix hands a lane four consecutive bytes of a
// row, so the MMA's k index (S^T = K Q^T) and M index (O^T = V^T P^T) are
// taken in a fixed permutation of the 16 dims of a step -- the query is loaded
// in the same permutation and the output rows are stored back in dim order.
// With kFused the kernel is the whole decode step (decode_step_paged_int8):
// each CTA normalises and rotates its query heads, the warp whose chunk holds
// position T-1 quantizes the new K and V rows, appends them and patches them
// into its staged chunk (as the bf16 fused step does), so every history chunk
// may be requested before griddepcontrol.wait.
// Per-key K scales multiply the scores; per-key V scales are folded into P,
// which is split into fp16 hi + lo parts. Partition states go to the
// workspace; the last CTA of a (sequence, KV head) to finish merges them
// (partition_merge.cuh), or merge_kernel does when they do not fit its
// shared memory.
#include <algorithm>
#include <cmath>

#include <cuda.h>

#include "common.cuh"
#include "head_norm_rope.cuh"
#include "launch.h"
#include "partition_merge.cuh"
#include "quantize_int8.cuh"
#include "tensor_map.h"

namespace pgqa {
namespace {

__device__ unsigned g_flags_int8;

__device__ __forceinline__ void raise_flag8(unsigned f) { atomicOr(&g_flags_int8, f); }

constexpr int kTile8 = kChunkTokens * 128;         // 16 rows x 128 int8 codes
constexpr int kStage8 = 2 * kTile8;                // K tile, V tile
constexpr int kScaleBytes8 = 2 * kChunkTokens * 4; // K scales, V scales
constexpr int kFusedMergeMax8 = 64;                // partitions the last CTA merges itself
// Partitions of at least this many chunks use the 16-warp shape.
constexpr int kDeepChunks8 = 64;

// CTA shapes: kW warps, each owning every kW-th chunk of its partition in a
// ring of kS stages folded kGroup at a time, kCtas CTAs per SM.
template <int kW, int kS, int kCtas, int kGrp = 0> struct Shape8 {
    static constexpr int kWarps = kW;
    static constexpr int kStages = kS;
    static constexpr int kCtasPerSm = kCtas;
    // chunks folded together: kGrp if given, else half the ring (one half
    // loads while the other folds), and at least a pair when the ring has
    // room for one
    static constexpr int kGroup = kGrp ? kGrp : (kStages >= 4 ? kStages / 2 : (kStages >= 2 ? 2 : 1));
    static constexpr int kStageArea = kWarps * kStages * kStage8;
    static constexpr int kScaleOffset = kStageArea;
    static constexpr int kBarOffset = kScaleOffset + kWarps * kStages * kScaleBytes8;
    static constexpr int kRowsOffset = kBarOffset + kWarps * kStages * 8;
    static constexpr int kTicketOffset = (kRowsOffset + kWarps * kStages * 4 + 7) & ~7;
    static constexpr int kMergeBarOffset = kTicketOffset + 8;
    // fused step: the rotated query [G][128] bf16, then the appended row as
    // it goes into its staged chunk (K codes, V codes [128] each, the K and V
    // scales)
    static constexpr int kQBufOffset = (kMergeBarOffset + 8 + 15) & ~15;
    static constexpr int kPatchOffset = kQBufOffset + kMaxGroup * kHeadDim * 2;
    static constexpr int kSmem = 1024 /* alignment slack */ + kPatchOffset + 2 * kHeadDim + 16;
    static constexpr int kMergeScratch = merge_scratch_bytes<kWarps * 32, kFusedMergeMax8>(kMaxGroup);
    // chunks per warp requested before griddepcontrol.wait: all of the ring
    // (the fused step on the T = 8192 chain with 9 warps x 6 stages: 9.11 us
    // per layer with all stages, 9.20 with 4, 9.32 with 3, 9.59 with 2)
    template <bool kFused> static constexpr int kPrewait = kStages;
    static_assert(kSmem <= 232448, "exceeds the 227 KiB of shared memory a CTA may hold");
    static_assert(kCtas * (kSmem + 1024) <= 233472, "228 KB of shared memory per SM, 1 KB reserved per CTA");
    static_assert(kGroup >= 1 && kGroup <= 3, "fold groups of 1 to 3 chunks");
};
// 12 warps x 3 stages for short partitions in one wave (the T = 8192 layer
// chain: up to 3 chunks per warp, all in flight at once). The chain's time
// after the query arrives is the fold of every chunk of the partition, which
// is issue-bound: three warps per SM sub-partition instead of 9 warps (one
// sub-partition with three, the others two) fold it sooner. 28-layer chain,
// same process: fused step 8.11 us per layer against 8.64 for 9 x 6 and
// 8.08 for 12 x 4 (attention alone 7.84, 8.34, 7.91); 3 stages take less
// shared memory than 4 for the same time.
using Shape8Short = Shape8<12, 3, 1>;
// Long partitions are bound by the fold's latency: a warp issues about once
// in 5.4 cycles (MMA and conversion chains), so the SM wants four warps on
// each of its sub-partitions, i.e. 16 warps (the most that fit 128
// registers a thread), each folding one chunk at a time while its other two
// stages load. B = 1, Hq = 32, T = 131072, 19 partitions, same process
// (us): 16 x 3 one at a time 45.7, 16 x 3 in pairs 48.2, 12 x 4 in pairs
// 50.6, 12 x 4 one at a time 52.2, 8 x 6 in threes 58.3, 20 x 2 (spills)
// 45.2.
using Shape8Deep = Shape8<16, 3, 1, 1>;
// Grids of several waves run several CTAs per SM, so that one CTA's start
// (table and context loads, first request) and end (merge, state write)
// overlap the others' streaming: four of 4 warps x 3 stages (about 52 KiB
// each) for partitions up to 1024 positions, two of 8 warps x 3 stages
// (about 104 KiB) otherwise; 16 warps per SM as above, each folding one
// chunk at a time. Two CTAs of 8 warps against one of 16 for longer
// partitions (us): B = 64 ragged contexts, 4096-position partitions 364.1
// against 398.4; B = 1, Hq = 32, T = 131072 with 2731-, 4096- and
// 5462-position partitions 60.3 / 52.3 / 67.8 against 61.8 / 57.5 / 70.8. B = 1, Hq = 32, T = 131072 (us, this
// shape / the earlier three of 4 x 4 or two of 6 x 4, in pairs): 512-position
// partitions 58.9 / 64.9, 1024 52.5 / 60.3, 2048 56.3 / 60.0; three of
// 4 x 4 one at a time 66.0 (512) and 62.5 (1024); 512-position partitions
// on two of 8 x 3: 67.8.
using Shape8Pair = Shape8<8, 3, 2, 1>;
using Shape8Quad = Shape8<4, 3, 4, 1>;
constexpr int kQuadMaxPositions8 = 1024;

struct Int8Params {
    const uint16_t *q;
    const int32_t *block_table, *context_lens;
    const float *k_scale, *v_scale;
    float *out_f32;
    uint16_t *out_bf16;
    float *ws_m, *ws_l, *ws_acc;
    unsigned *tickets; // [B*Hkv] partition tickets (in-kernel merge)
    int Hq, Hkv, P, max_pages, num_pages, NP, ppp;
    int fused_merge;
    // 1: tmap_k spans both code caches (one TMA load per chunk's K and V
    // tiles); 1: tmap_s spans both scale arrays (one load per chunk's scales)
    int kv_map, scale_map;
    float scale_log2;
    // fused decode step only: the new token's raw heads, the prologue's
    // parameters and the cache to append to
    const uint16_t *q_raw, *k_new, *v_new, *gamma_q, *gamma_k;
    int8_t *k_cache8, *v_cache8;
    float *k_scale_out, *v_scale_out;
    uint16_t *q_out;
    float eps;
    RopeFreqs freqs;
#ifdef PGQA_TIMELINE
    unsigned long long *tl; // timeline buffer, or NULL
    int tl_launch;          // this launch's index in it
#endif
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
    template <int NC, int NG>
    __device__ __forceinline__ void fold(const uint32_t (&stage)[NG], const float *const (&scl)[NG],
                                         const int (&rows)[NG], float scale_log2)
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

template <int G, bool kFused, typename S>
__global__ void __launch_bounds__(S::kWarps * 32, S::kCtasPerSm)
    decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_s, const Int8Params p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

    allow_dependent_launch();
    TL_STAMP(0);
    unsigned char *stages = smem + warp * S::kStages * kStage8;
    float *scales = reinterpret_cast<float *>(smem + S::kScaleOffset) + warp * S::kStages * 2 * kChunkTokens;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBarOffset) + warp * S::kStages;
    int *stage_rows = reinterpret_cast<int *>(smem + S::kRowsOffset) + warp * S::kStages;
    if (lane == 0) {
        if (warp == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            prefetch_tensormap(&tmap_s);
        }
#pragma unroll
        for (int s = 0; s < S::kStages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }

    const int part_tokens = p.ppp * p.P;
    const int tok0 = part * part_tokens;
    const int32_t *table = p.block_table + static_cast<size_t>(b) * p.max_pages;
    auto chunk_token = [&](int k) { return tok0 + (warp + k * S::kWarps) * kChunkTokens; };
    // The first 32 table entries of this warp's chunks are loaded before the
    // context length is known (any entry below max_pages may be read), both
    // loads issued where they stand, so the first requests wait for one
    // memory round trip, not two.
    int tbl_blk = 0, tbl_val = -1;
    {
        const int page = chunk_token(lane) / p.P;
        if (chunk_token(lane) < tok0 + part_tokens && page < p.max_pages)
            tbl_val = ldg_i32_now(table + page);
    }
    int T = ldg_i32_now(p.context_lens + b);
    if (T < (kFused ? 1 : 0) || T > p.max_pages * p.P) {
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
    const int my_chunks = (n_chunks > warp) ? (n_chunks - 1 - warp) / S::kWarps + 1 : 0;
    __syncwarp();

    // the chunk holding position T-1 is written by the prologue this kernel
    // may overlap: it is requested after griddepcontrol.wait (the fused step
    // patches the new row into shared memory itself instead)
    auto holds_new_token = [&](int k) { return !kFused && chunk_token(k) + kChunkTokens > T - 1; };
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
    auto issue = [&](int k, int phys, uint64_t policy) { // lane 0
        const int t = chunk_token(k);
        uint64_t *bar = &bars[k % S::kStages];
        if (phys < 0 || phys >= p.num_pages) {
            raise_flag8(PGQA_DEVERR_BAD_PAGE);
            stage_rows[k % S::kStages] = 0;
            mbar_arrive(bar);
            return;
        }
        stage_rows[k % S::kStages] = min(kChunkTokens, tok1 - t);
        const int row = (phys * p.Hkv + kvh) * p.P + (t % p.P);
        unsigned char *dst = stages + (k % S::kStages) * kStage8;
        float *sdst = scales + (k % S::kStages) * 2 * kChunkTokens;
        mbar_arrive_expect_tx(bar, kStage8 + kScaleBytes8);
        if (p.kv_map) {
            tma_load_3d(dst, &tmap_k, 0, row, 0, bar, policy);
        } else {
            tma_load_2d(dst, &tmap_k, 0, row, bar, policy);
            tma_load_2d(dst + kTile8, &tmap_v, 0, row, bar, policy);
        }
        if (p.scale_map) {
            tma_load_2d(sdst, &tmap_s, row, 0, bar, policy);
        } else {
            bulk_copy_g2s(sdst, p.k_scale + row, kChunkTokens * 4, bar, policy);
            bulk_copy_g2s(sdst + kChunkTokens, p.v_scale + row, kChunkTokens * 4, bar, policy);
        }
    };

    const uint64_t policy = l2_evict_first_policy();
    const int first = min(S::kStages, my_chunks);
    int first_phys[S::kStages];
#pragma unroll
    for (int k = 0; k < S::kStages; ++k)
        first_phys[k] = k < first ? phys_of(k) : -1;
    TL_STAMP(1);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < S::kStages; ++k)
            if (k < first && k < S::template kPrewait<kFused> && !holds_new_token(k))
                issue(k, first_phys[k], policy);
    }
    TL_STAMP(2);

    // fused step: warps < G rotate the query heads; the warp owning the chunk
    // of position T-1 quantizes and appends the new K and V rows. What no
    // earlier kernel writes (gains, rotation, the append slot) is prepared
    // before the wait.
    const int pos = T - 1;
    const bool has_q = kFused && T > 0 && warp < G;
    int new_chunk = -1, new_phys = -1;
    if (kFused && T > 0 && pos >= tok0 && pos < tok1) {
        const int c_idx = (pos - tok0) / kChunkTokens;
        if (c_idx % S::kWarps == warp) {
            new_chunk = c_idx / S::kWarps;
            new_phys = table[pos / p.P];
        }
    }
    HeadRope rope;
    float gain_q[4], gain_k[4];
    if (has_q || new_chunk >= 0)
        rope.init(pos, p.freqs);
    if (has_q)
        load_head(p.gamma_q, gain_q);
    if (new_chunk >= 0)
        load_head(p.gamma_k, gain_k);

    grid_dependency_wait();
    TL_STAMP(3);

    const size_t row0 = static_cast<size_t>(b) * p.Hq + kvh * G;
    const size_t krow = (static_cast<size_t>(b) * p.Hkv + kvh) * kHeadDim;
    float xq[4], xk[4], xv[4];
    if (has_q)
        load_head(p.q_raw + (row0 + warp) * kHeadDim, xq);
    if (new_chunk >= 0) {
        load_head(p.k_new + krow, xk);
        load_head(p.v_new + krow, xv);
    }
    Int8Warp<G> st;
    if constexpr (!kFused)
        st.init(p.q + row0 * kHeadDim);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < S::kStages; ++k)
            if (k < first && (k >= S::template kPrewait<kFused> || holds_new_token(k)))
                issue(k, first_phys[k], policy);
    }
    __syncwarp();

    // fused step: normalise and rotate q; once every warp has its query, the
    // warp owning the new position normalises and rotates K, quantizes K (its
    // bf16 rounding) and V, appends them and keeps the row in shared memory
    // for the patch of its staged chunk.
    unsigned char *patch = smem + S::kPatchOffset;
    if constexpr (kFused) {
        uint16_t *q_buf = reinterpret_cast<uint16_t *>(smem + S::kQBufOffset);
        if (has_q) {
            norm_rope_apply(xq, gain_q, p.eps, rope);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint16_t bits = f32_to_bf16_bits(xq[i]);
                q_buf[warp * kHeadDim + lane + 32 * i] = bits;
                if (part == 0 && p.q_out)
                    p.q_out[(row0 + warp) * kHeadDim + lane + 32 * i] = bits;
            }
        }
        __syncthreads();
        st.init(q_buf);
        TL_STAMP(4);
        if (new_chunk >= 0) {
            int kc[4], vc[4];
            norm_rope_apply(xk, gain_k, p.eps, rope);
            round_head_bf16(xk);
            const float ks = quantize_head_int8(xk, kc);
            const float vs = quantize_head_int8(xv, vc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                patch[lane + 32 * i] = static_cast<unsigned char>(kc[i]);
                patch[kHeadDim + lane + 32 * i] = static_cast<unsigned char>(vc[i]);
            }
            if (lane == 0) {
                reinterpret_cast<float *>(patch + 2 * kHeadDim)[0] = ks;
                reinterpret_cast<float *>(patch + 2 * kHeadDim)[1] = vs;
            }
            if (new_phys >= 0 && new_phys < p.num_pages) {
                const size_t slot_row = (static_cast<size_t>(new_phys) * p.Hkv + kvh) * p.P + pos % p.P;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p.k_cache8[slot_row * kHeadDim + lane + 32 * i] = static_cast<int8_t>(kc[i]);
                    p.v_cache8[slot_row * kHeadDim + lane + 32 * i] = static_cast<int8_t>(vc[i]);
                }
                if (lane == 0) {
                    p.k_scale_out[slot_row] = ks;
                    p.v_scale_out[slot_row] = vs;
                }
            } else if (lane == 0) {
                raise_flag8(PGQA_DEVERR_BAD_PAGE);
            }
            __syncwarp();
        }
    }

    bool ok = true;
    int k0 = 0;
    // As in the bf16 kernel: pairs for warps with few chunks, whole groups
    // otherwise (the grouping depends only on the chunk count).
    const int group = min(S::kGroup, my_chunks <= 2 * S::kGroup ? 2 : S::kGroup);
    for (int nc; k0 < my_chunks; k0 += nc) {
        nc = min(group, my_chunks - k0);
        uint32_t stage_addr[S::kGroup];
        const float *scl[S::kGroup];
        int rows[S::kGroup];
#pragma unroll
        for (int c = 0; c < S::kGroup; ++c) {
            const int k = k0 + c;
            stage_addr[c] = smem_addr(stages + (k % S::kStages) * kStage8);
            scl[c] = scales + (k % S::kStages) * 2 * kChunkTokens;
            rows[c] = 0;
            if (c < nc) {
                const bool landed = mbar_wait_bounded(&bars[k % S::kStages], (k / S::kStages) & 1);
                if (!__all_sync(0xFFFFFFFFu, landed))
                    ok = false;
                if (k == 1)
                    TL_STAMP(5);
                if (k == my_chunks - 1)
                    TL_STAMP_LATEST(6);
                rows[c] = stage_rows[k % S::kStages];
                if (kFused && k == new_chunk && rows[c] > 0) {
                    // the staged copy predates the append: put the new row in
                    // (word w < 64 of the patch: bytes 4w..4w+3 of the K row,
                    // then of the V row)
                    const int r = pos % kChunkTokens;
                    unsigned char *stage = stages + (k % S::kStages) * kStage8;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int w = lane + 32 * i, x = 4 * (w & 31);
                        const int off = (w >> 5) * kTile8 + r * 128 + (((x >> 4) ^ (r & 7)) << 4) + (x & 15);
                        *reinterpret_cast<uint32_t *>(stage + off) = reinterpret_cast<const uint32_t *>(patch)[w];
                    }
                    if (lane < 2)
                        scales[(k % S::kStages) * 2 * kChunkTokens + lane * kChunkTokens + r] =
                            reinterpret_cast<const float *>(patch + 2 * kHeadDim)[lane];
                    __syncwarp();
                }
            }
        }
        if (!ok)
            break;
        if (S::kGroup >= 3 && nc == 3)
            st.template fold<(S::kGroup >= 3 ? 3 : 1)>(stage_addr, scl, rows, p.scale_log2);
        else if (S::kGroup >= 2 && nc == 2)
            st.template fold<(S::kGroup >= 2 ? 2 : 1)>(stage_addr, scl, rows, p.scale_log2);
        else
            st.template fold<1>(stage_addr, scl, rows, p.scale_log2);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < S::kGroup; ++c) {
            const int k = k0 + c + S::kStages;
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
        const int issued = min(my_chunks, k0 + S::kStages);
        for (int kk = k0; kk < issued; ++kk)
            (void)mbar_wait_bounded(&bars[kk % S::kStages], (kk / S::kStages) & 1);
        st.clear();
    }
    __syncwarp();
    // every copy into this warp's stages has landed: they can hold its record
    st.store_record(reinterpret_cast<float *>(stages));
    __syncthreads();
    TL_STAMP(7);

    for (int e = threadIdx.x; e < G * kHeadDim; e += S::kWarps * 32) {
        const int h = e / kHeadDim, d = e % kHeadDim;
        float M = kEmptyMax;
#pragma unroll
        for (int w = 0; w < S::kWarps; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * S::kStages * kStage8);
            M = fmaxf(M, rec[G * kHeadDim + h]);
        }
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < S::kWarps; ++w) {
            const float *rec = reinterpret_cast<const float *>(smem + w * S::kStages * kStage8);
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
    if (n_parts == 1 || !p.fused_merge)
        return;

    // Ticket: the CTA that finishes last for this (sequence, KV head) merges.
    // The barrier orders every thread's partial-state stores before thread
    // 0's release; its acquire (when last) orders the other CTAs' stores
    // before the merge's loads, which the second barrier extends to all
    // threads.
    unsigned *ticket_slot = reinterpret_cast<unsigned *>(smem + S::kTicketOffset);
    TL_STAMP(8);
    __syncthreads();
    unsigned *ticket = p.tickets + static_cast<size_t>(b) * p.Hkv + kvh;
    if (threadIdx.x == 0)
        *ticket_slot = atomic_add_acq_rel_gpu(ticket, 1u);
    __syncthreads();
    TL_STAMP(9);
    if (*ticket_slot != static_cast<unsigned>(n_parts - 1))
        return;
    const auto row_of = [&](int c) { return row0 + c; };
    if (!merge_partitions_in_cta<G, S::kWarps * 32, kFusedMergeMax8>(
            p.ws_m, p.ws_l, p.ws_acc, p.NP, n_parts, row_of, p.out_f32, p.out_bf16, smem,
            reinterpret_cast<uint64_t *>(smem + S::kMergeBarOffset)) &&
        threadIdx.x == 0)
        raise_flag8(PGQA_DEVERR_WAIT_TIMEOUT); // the merge's copy never landed: outputs left alone
#ifdef PGQA_TIMELINE
    __syncthreads();
    TL_STAMP(10);
#endif
    if (threadIdx.x == 0)
        *ticket = 0u; // ready for the next call
}

// An INT8 cache as a 2-D tensor [rows][128 bytes]; one box {128, 16} is a
// 16-row tile with 128-byte swizzle.
cudaError_t encode_int8_map(CUtensorMap *map, const void *base, long long rows)
{
    EncodeTiledFn fn = tensor_map_encoder();
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

// Both code caches as one 3-D tensor [2 caches][rows][128 bytes] (the
// outer dimension steps from k_cache8 to v_cache8): one box {128, 16, 2}
// lands a chunk's K tile and V tile (128-byte swizzle) with one TMA
// instruction. Needs v_cache8 above k_cache8 by a multiple of 16 bytes.
cudaError_t encode_int8_kv_map(CUtensorMap *map, const void *k_base, const void *v_base, long long rows)
{
    const uintptr_t k = reinterpret_cast<uintptr_t>(k_base), v = reinterpret_cast<uintptr_t>(v_base);
    if (v <= k || (v - k) % 16 != 0 || v - k >= (1ull << 40))
        return cudaErrorInvalidValue;
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(rows), 2u};
    const cuuint64_t strides[2] = {128u, static_cast<cuuint64_t>(v - k)};
    const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(kChunkTokens), 2u};
    const cuuint32_t elem[3] = {1u, 1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(k_base), dims, strides, box,
                          elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Both scale arrays as one 2-D tensor [2 arrays][rows] fp32: one box
// {16, 2} lands a chunk's 16 K scales and 16 V scales. Needs v_scale above
// k_scale by a multiple of 16 bytes.
cudaError_t encode_scale_map(CUtensorMap *map, const float *k_scale, const float *v_scale, long long rows)
{
    const uintptr_t k = reinterpret_cast<uintptr_t>(k_scale), v = reinterpret_cast<uintptr_t>(v_scale);
    if (v <= k || (v - k) % 16 != 0 || v - k >= (1ull << 40))
        return cudaErrorInvalidValue;
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), 2u};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(v - k)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkTokens), 2u};
    const cuuint32_t elem[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(k_scale), dims, strides, box,
                          elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int G, bool kFused, typename S>
cudaError_t launch_int8_t(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &ms,
                          const Int8Params &kp, dim3 grid, cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 64 || !configured[dev]) {
        err = cudaFuncSetAttribute(decode_int8_kernel<G, kFused, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   S::kSmem);
        if (err != cudaSuccess)
            return err;
        if (dev < 64)
            configured[dev] = true;
    }
    return launch_pdl(decode_int8_kernel<G, kFused, S>, grid, dim3(S::kWarps * 32), S::kSmem, stream, mk, mv, ms,
                      kp);
}

template <typename S> bool merges_in_kernel(int G, int num_partitions)
{
    return num_partitions <= kFusedMergeMax8 &&
           static_cast<long>(G) * num_partitions * kHeadDim * 4 + S::kMergeScratch <= S::kStageArea;
}

enum class Shape8Kind { kShort, kDeep, kPair, kQuad };

template <int G>
cudaError_t launch_int8_g(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &ms,
                          const Int8Params &kp, dim3 grid, bool fused, Shape8Kind shape, cudaStream_t stream)
{
    if constexpr (G <= Shape8Quad::kWarps) {
        if (shape == Shape8Kind::kQuad)
            return fused ? launch_int8_t<G, true, Shape8Quad>(mk, mv, ms, kp, grid, stream)
                         : launch_int8_t<G, false, Shape8Quad>(mk, mv, ms, kp, grid, stream);
    }
    if constexpr (G <= Shape8Pair::kWarps) {
        if (shape == Shape8Kind::kPair)
            return fused ? launch_int8_t<G, true, Shape8Pair>(mk, mv, ms, kp, grid, stream)
                         : launch_int8_t<G, false, Shape8Pair>(mk, mv, ms, kp, grid, stream);
    }
    if (shape == Shape8Kind::kDeep)
        return fused ? launch_int8_t<G, true, Shape8Deep>(mk, mv, ms, kp, grid, stream)
                     : launch_int8_t<G, false, Shape8Deep>(mk, mv, ms, kp, grid, stream);
    return fused ? launch_int8_t<G, true, Shape8Short>(mk, mv, ms, kp, grid, stream)
                 : launch_int8_t<G, false, Shape8Short>(mk, mv, ms, kp, grid, stream);
}

} // namespace

cudaError_t launch_decode_int8(const DecodeInt8Args &a, cudaStream_t stream)
{
    if (a.B == 0)
        return cudaSuccess;
    const int G = a.Hq / a.Hkv;
    CUtensorMap mk, mv, ms;
    const long long rows = static_cast<long long>(a.num_pages) * a.Hkv * a.page_size;
    if (rows == 0)
        return cudaErrorInvalidValue;
    Int8Params kp{};
    cudaError_t err = encode_int8_kv_map(&mk, a.k_cache8, a.v_cache8, rows);
    if (err == cudaSuccess) {
        kp.kv_map = 1;
        mv = mk;
    } else {
        err = encode_int8_map(&mk, a.k_cache8, rows);
        if (err == cudaSuccess)
            err = encode_int8_map(&mv, a.v_cache8, rows);
        if (err != cudaSuccess)
            return err;
    }
    if (encode_scale_map(&ms, a.k_scale, a.v_scale, rows) == cudaSuccess)
        kp.scale_map = 1;
    else
        ms = mk; // unused

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
#ifdef PGQA_TIMELINE
    kp.tl = timeline_buffer();
    kp.tl_launch = timeline_next_launch();
#endif
    if (a.fused) {
        kp.q_raw = a.q_raw;
        kp.k_new = a.k_new;
        kp.v_new = a.v_new;
        kp.gamma_q = a.gamma_q;
        kp.gamma_k = a.gamma_k;
        kp.k_cache8 = const_cast<int8_t *>(a.k_cache8);
        kp.v_cache8 = const_cast<int8_t *>(a.v_cache8);
        kp.k_scale_out = const_cast<float *>(a.k_scale);
        kp.v_scale_out = const_cast<float *>(a.v_scale);
        kp.q_out = a.q_out;
        kp.eps = a.eps;
        kp.freqs = make_rope_freqs(a.rope_theta);
    }
    // Grids of more than one wave (of one CTA per SM) take four (short
    // partitions) or two CTAs per SM (the fused step and attention alone
    // alike, so they give equal bits); one-wave grids take 16 warps x 3
    // stages for long partitions, 12 warps x 3 for short ones (both
    // fold-bound).
    const long part_positions = static_cast<long>(a.pages_per_part) * a.page_size;
    const bool waves = a.num_partitions > 1 &&
                       static_cast<long>(a.B) * a.Hkv * a.num_partitions > (a.sm_count > 0 ? a.sm_count : 1);
    Shape8Kind shape = part_positions >= kDeepChunks8 * kChunkTokens ? Shape8Kind::kDeep : Shape8Kind::kShort;
    if (waves && G <= Shape8Quad::kWarps && part_positions <= kQuadMaxPositions8)
        shape = Shape8Kind::kQuad;
    else if (waves && G <= Shape8Pair::kWarps)
        shape = Shape8Kind::kPair;
    const bool in_kernel = shape == Shape8Kind::kQuad   ? merges_in_kernel<Shape8Quad>(G, a.num_partitions)
                           : shape == Shape8Kind::kPair ? merges_in_kernel<Shape8Pair>(G, a.num_partitions)
                           : shape == Shape8Kind::kDeep ? merges_in_kernel<Shape8Deep>(G, a.num_partitions)
                                                        : merges_in_kernel<Shape8Short>(G, a.num_partitions);
    kp.fused_merge = in_kernel ? 1 : 0;
    if (a.num_partitions > 1) {
        const size_t n = static_cast<size_t>(a.B) * a.Hq * a.num_partitions;
        const auto align256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
        char *ws = reinterpret_cast<char *>(a.ws);
        kp.tickets = reinterpret_cast<unsigned *>(ws);
        ws += decode_ticket_bytes(a.B, a.Hkv);
        kp.ws_m = reinterpret_cast<float *>(ws);
        kp.ws_l = reinterpret_cast<float *>(ws + align256(n * sizeof(float)));
        kp.ws_acc = reinterpret_cast<float *>(ws + 2 * align256(n * sizeof(float)));
    }
    const dim3 grid(a.num_partitions, a.Hkv, a.B);
    switch (G) {
    case 1: err = launch_int8_g<1>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 2: err = launch_int8_g<2>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 3: err = launch_int8_g<3>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 4: err = launch_int8_g<4>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 5: err = launch_int8_g<5>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 6: err = launch_int8_g<6>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 7: err = launch_int8_g<7>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    case 8: err = launch_int8_g<8>(mk, mv, ms, kp, grid, a.fused, shape, stream); break;
    default: return cudaErrorInvalidValue;
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
    ma.out_f32 = a.out_f32;
    ma.out_bf16 = a.out_bf16;
    ma.context_lens = a.context_lens;
    ma.page_size = a.page_size;
    ma.pages_per_part = a.pages_per_part;
    ma.max_pages = a.max_pages;
    return launch_merge(ma, stream);
}

// Same layout as the bf16 kernel's workspace: partition tickets [B*Hkv]
// (zero before first use; every completed call leaves them zero), then m, l
// [B*Hq*NP] and acc [B*Hq*NP*128].
size_t decode_int8_workspace_bytes(int B, int Hkv, int Hq, int num_partitions)
{
    return decode_workspace_bytes(B, Hkv, Hq, num_partitions);
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
