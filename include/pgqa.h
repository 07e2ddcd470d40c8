/*
 * pgqa.h -- C ABI of the paged GQA decode-attention library (libpgqa.so),
 * sm_103a (GB300).
 *
 * The library computes the single-token decode step of grouped-query
 * attention over a paged bf16 KV cache:
 *   - the fused prologue: per-head Q/K RMSNorm, half-rotation RoPE and the
 *     append of the new token's K/V into the paged cache;
 *   - decode attention with (m, l, acc) online softmax, split over KV
 *     partitions and merged exactly;
 *   - both in one launch per layer (decode_step_paged);
 *   - a host-tiled variant that keeps (m, l, acc) in global memory while KV
 *     tiles are streamed in from pinned host memory, and a zero-copy variant
 *     that reads a history held in pinned host memory directly.
 *
 * Sources (page title, section):
 *   "From Qwen3 math to CUDA kernels: a 0.6B inference runtime"
 *       s2.1 RMSNorm, s2.3 Q/K head RMSNorm, s2.4 RoPE, s2.5 GQA head map,
 *       s2.6 scaled dot-product attention (causal), s5.1 current stream,
 *       s5.2 no allocation on the hot path, s7.1 one warp per head,
 *       s7.2 logical token -> physical cache address, s9.1 exact partition
 *       merge, s10.1 grouped single-CTA path, s10.2 partitioned path.
 *   "EdgeTransformerEngine"
 *       online-softmax note (state (m, l, acc) and its update step),
 *       KV-offload design (attn_init / attn_tile / attn_finalize kernels,
 *       512-position tiles, m = -1e30), copy/compute stream events.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Types. pgqa_bf16 is a bf16 bit pattern (the top half of a binary32).
 *   All float state is IEEE binary32. Index arrays are int32.
 * Shapes. D (head dimension) must be 128. Hq % Hkv == 0 and the group size
 *   g = Hq / Hkv must lie in [1, 8]. Query head h reads KV head h / g.
 * Cache layout. k_cache and v_cache are [num_pages][Hkv][page_size][D] bf16:
 *   the rows of one (physical page, KV head) are contiguous. Position pos of
 *   sequence b lives in physical page block_table[b * max_pages + pos /
 *   page_size] at in-page offset pos % page_size. page_size is a power of two
 *   in [16, 256].
 * Context lengths. context_lens[b] = T_b counts the new token, which sits at
 *   position T_b - 1 and attends to all T_b positions (itself included).
 * Memory. Every pointer is caller-owned device memory unless stated
 *   otherwise; the library never allocates or frees memory. Tensor pointers
 *   (bf16 and float arrays) must be 16-byte aligned; index arrays 4-byte.
 * Streams. All work is enqueued on the stream the caller passes; nothing is
 *   synchronised and the default stream is never used implicitly. Calls are
 *   capturable into CUDA graphs except pgqa_device_error (synchronous).
 * Errors. Every call returns PGQA_OK (0) or a negative PGQA_ERR_* code and
 *   never throws; pgqa_last_error() returns the calling thread's message for
 *   its last failing call. Invalid data that only the device can see (a
 *   block-table entry outside [0, num_pages), a context length above
 *   max_pages * page_size) never causes an out-of-bounds access: the
 *   affected keys or slots are skipped and a sticky per-device flag is
 *   raised, readable with pgqa_device_error().
 */
#ifndef PGQA_H
#define PGQA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pgqa_bf16;

enum pgqa_status {
    PGQA_OK = 0,
    PGQA_ERR_INVALID_ARG = -1, /* null pointer, negative size, inconsistent shapes */
    PGQA_ERR_UNSUPPORTED = -2, /* D != 128, g outside [1, 8], page_size not in {16..256} */
    PGQA_ERR_MISALIGNED = -3,  /* a tensor pointer is not 16-byte aligned */
    PGQA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
    PGQA_ERR_CUDA = -5         /* a CUDA runtime call or launch failed */
};

/* Sticky device-side flags (bit mask) read by pgqa_device_error(). */
#define PGQA_DEVERR_BAD_PAGE 1u     /* block-table entry outside [0, num_pages) */
#define PGQA_DEVERR_BAD_CONTEXT 2u  /* context length < 0 (or < 1 for the prologue) or too long */
#define PGQA_DEVERR_WAIT_TIMEOUT 4u /* a bounded wait (an asynchronous copy) ran out */

/* Message of the calling thread's last failing call ("" if none). */
const char *pgqa_last_error(void);

/* Read the sticky device flags of the current device into *flags_out (OR of
 * PGQA_DEVERR_*) and clear them if clear != 0. Synchronises the device. */
int pgqa_device_error(unsigned *flags_out, int clear);

/*
 * pgqa_selftest_wait_timeout -- exercises the library's failure path for a
 * wait that never completes (no counterpart on the pages): one CTA waits on
 * an mbarrier that nothing arrives on; the wait gives up after its limit
 * (200 ms), the kernel raises PGQA_DEVERR_WAIT_TIMEOUT and returns, and the
 * context stays usable. Enqueued on `stream`; read the flag with
 * pgqa_device_error. Every wait in the library's kernels is bounded the same
 * way.
 */
int pgqa_selftest_wait_timeout(cudaStream_t stream);

/*
 * qk_norm_rope_append -- fused decode prologue for one layer.
 * Follows s2.3 (per-head RMSNorm with learned gains, eps), s2.4 (RoPE on the
 * pairs (i, i + D/2), omega_i = theta^(-2i/D), phase pos * omega_i), s7.1
 * (one warp per head) and s7.2 (write the rotated K straight into its
 * physical page).
 *
 *   q       [B][Hq][D]  bf16   new token's query heads
 *   k, v    [B][Hkv][D] bf16   new token's key / value heads
 *   gamma_q, gamma_k [D] bf16  RMSNorm gains (shared by all heads)
 *   context_lens [B] int32     T_b >= 1; the new token sits at pos = T_b - 1
 *   block_table [B][max_pages] int32
 *   k_cache, v_cache           paged cache (layout above); only the slots
 *                              (b, h, pos) are written: K = bf16(RoPE(RMSNorm(k))),
 *                              V = v bit for bit
 *   q_out   [B][Hq][D]  bf16   bf16(RoPE(RMSNorm(q)))
 * Arithmetic in fp32; the RoPE phase is formed and reduced in fp64 so that it
 * stays accurate at large positions. bf16 results are rounded to nearest even.
 * A sequence with an invalid T_b or page is skipped (flag raised).
 */
int qk_norm_rope_append(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                        const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                        const int32_t *context_lens, const int32_t *block_table,
                        pgqa_bf16 *k_cache, pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq,
                        int Hkv, int D, int page_size, int max_pages, int num_pages,
                        float rope_theta, float eps, cudaStream_t stream);

/*
 * decode_attn_partition_count -- number of KV partitions NP that
 * decode_attn_paged will use for these arguments (num_partitions = 0 picks
 * one from the current device's SM count; otherwise it is clamped to
 * [1, max_pages]). Each partition covers ceil(max_pages / NP) pages.
 */
int decode_attn_partition_count(int B, int Hkv, int page_size, int max_pages,
                                int num_partitions);

/*
 * decode_attn_workspace_size -- bytes of device workspace decode_attn_paged
 * needs (0 when NP = 1). Same arguments as decode_attn_paged; the auto
 * choice depends on the current device.
 */
size_t decode_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                  int num_partitions);

/*
 * decode_attn_paged -- causal GQA decode attention over the paged cache.
 * Follows s2.5/s2.6 (query head h attends with KV head h/g over positions
 * 0 .. T_b - 1: s_j = scale * <q_h, K_j>, softmax, weighted sum of V_j),
 * the online-softmax update of the (m, l, acc) state, s10.1 (one CTA serves
 * all g query heads of a KV head and reads each K/V tile once), s10.2 and
 * s9.1 (the history is split into NP partitions whose states are merged
 * exactly: M = max m_p, out = sum_p acc_p e^(m_p - M) / sum_p l_p e^(m_p - M)).
 *
 *   q            [B][Hq][D] bf16 (the prologue's q_out)
 *   out_f32      [B][Hq][D] float, nullable
 *   out_bf16     [B][Hq][D] bf16 (nearest-even cast of the fp32 result), nullable
 *   workspace    device scratch of ws_bytes >= decode_attn_workspace_size(...)
 *                (may be NULL when that size is 0). Zero-fill it before the
 *                first call with given (B, Hq, Hkv, num_partitions, page_size,
 *                max_pages); every call that completes leaves it ready for
 *                the next call with the same arguments (its partition
 *                tickets back at zero). Calls whose work may overlap on the
 *                GPU must not share a workspace.
 * Launch and ordering: the kernels are launched with programmatic stream
 * serialisation. The attention kernel may start before the previous kernel
 * in the stream has finished and then already reads block_table,
 * context_lens and the cache rows of positions below T_b - 1; only q and the
 * row of position T_b - 1 (written by qk_norm_rope_append) are read after
 * that kernel completes. The previous kernel must therefore not write those
 * inputs (qk_norm_rope_append does not).
 *   num_partitions  0 = automatic, else the requested NP.
 * A sequence with T_b = 0 produces zeros. For given arguments on a given
 * device the results are reproducible bit for bit: the partition count, the
 * kernel's CTA shape (one CTA per SM, or two smaller ones for grids of more
 * than one wave whose partitions are at most 2048 positions) and every
 * summation order depend only on them and on the device's SM count. Up to
 * 64 partitions whose states fit the CTA's shared memory are merged by the
 * last CTA of each (sequence, KV head); otherwise a merge kernel follows in
 * the same stream. Grids of the two-CTA shape merged that way with few
 * (sequence, KV head) pairs run each CTA over a run of consecutive
 * partitions; the partition states, and so the results, are those of the
 * two-CTA shape, bit for bit.
 */
int decode_attn_paged(const pgqa_bf16 *q, const pgqa_bf16 *k_cache, const pgqa_bf16 *v_cache,
                      const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages, int num_pages, float scale,
                      int num_partitions, float *out_f32, pgqa_bf16 *out_bf16, void *workspace,
                      size_t ws_bytes, cudaStream_t stream);

/*
 * decode_step_paged -- one layer's whole decode step in one launch:
 * qk_norm_rope_append (s2.3, s2.4, s7.2) followed by decode_attn_paged
 * (s2.5, s2.6, s9.1, s10.1, s10.2), with the same results as calling the two
 * in order. Each attention CTA normalises and rotates the query heads it
 * serves; the CTA whose partition holds the new position appends the new
 * token's K and V to the cache. Fusing removes a launch and a dependency from
 * the per-layer chain, and lets every history chunk be requested before the
 * previous kernel in the stream finishes.
 *
 *   q, k, v, gamma_q, gamma_k, context_lens (T_b >= 1), block_table,
 *   k_cache, v_cache, rope_theta, eps     as for qk_norm_rope_append
 *   q_out    [B][Hq][D] bf16, nullable: the rotated query, if wanted
 *   scale, num_partitions, out_f32, out_bf16, workspace, ws_bytes
 *                                        as for decode_attn_paged
 * Sequences with T_b < 1 raise PGQA_DEVERR_BAD_CONTEXT and produce zeros.
 */
int decode_step_paged(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                      const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                      const int32_t *context_lens, const int32_t *block_table, pgqa_bf16 *k_cache,
                      pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D,
                      int page_size, int max_pages, int num_pages, float rope_theta, float eps,
                      float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                      void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Multi-query decode: M >= 1 new tokens per sequence decoded in one step
 * (speculative or multi-token-prediction verification). Token i (0 <= i < M)
 * of sequence b sits at position T_b - M + i, where context_lens[b] = T_b
 * counts all M new tokens, and attends causally to positions
 * 0 .. T_b - M + i: the same s2.6 attention as decode_attn_paged, once per
 * new token, with each token's own prefix. M = 1 is exactly the
 * single-token step.
 *
 * qk_norm_rope_append_multi -- the prologue for M tokens: as
 *   qk_norm_rope_append with q [B][M][Hq][D], k, v [B][M][Hkv][D] and q_out
 *   [B][M][Hq][D]; token i is rotated at position T_b - M + i and appended to
 *   its slot. Needs T_b >= M (else the sequence is skipped, flag raised).
 *   1 <= M <= 64.
 * decode_attn_paged_multi -- the attention for M tokens: q [B][M][Hq][D] (the
 *   prologue's q_out), out_f32 / out_bf16 [B][M][Hq][D]; other arguments as
 *   decode_attn_paged. One CTA serves the M x g (token, head) pairs of a KV
 *   head, so M * (Hq / Hkv) <= 8 (else PGQA_ERR_UNSUPPORTED). Sequences with
 *   T_b < M produce zeros (flag raised). The attention kernel reads the
 *   cache rows of positions below T_b - M before the previous kernel in the
 *   stream completes (programmatic serialisation), the M new rows after.
 * decode_attn_multi_workspace_size -- workspace bytes for the same arguments.
 */
int qk_norm_rope_append_multi(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                              const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                              const int32_t *context_lens, const int32_t *block_table,
                              pgqa_bf16 *k_cache, pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int M,
                              int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                              float rope_theta, float eps, cudaStream_t stream);
/*
 * decode_step_paged_multi -- qk_norm_rope_append_multi followed by
 *   decode_attn_paged_multi in one launch (as decode_step_paged for M = 1):
 *   q [B][M][Hq][D], k, v [B][M][Hkv][D], q_out (nullable) and outputs
 *   [B][M][Hq][D], M * (Hq / Hkv) <= 8, T_b >= M; workspace as
 *   decode_attn_multi_workspace_size. Each attention CTA rotates the (token,
 *   head) queries it serves; the CTA whose range holds a new position appends
 *   that token's K and V and requests the chunk holding it only afterwards.
 */
int decode_step_paged_multi(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                            const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                            const int32_t *context_lens, const int32_t *block_table, pgqa_bf16 *k_cache,
                            pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int M, int Hq, int Hkv, int D,
                            int page_size, int max_pages, int num_pages, float rope_theta, float eps,
                            float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                            void *workspace, size_t ws_bytes, cudaStream_t stream);
size_t decode_attn_multi_workspace_size(int B, int M, int Hq, int Hkv, int D, int page_size,
                                        int max_pages, int num_partitions);
int decode_attn_paged_multi(const pgqa_bf16 *q, const pgqa_bf16 *k_cache, const pgqa_bf16 *v_cache,
                            const int32_t *block_table, const int32_t *context_lens, int B, int M,
                            int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                            float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                            void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * INT8 KV cache (the quantization scheme of "From Qwen3 math to CUDA
 * kernels", s0.1 -- INT8 values times an FP32 scale, accumulated in FP32 --
 * and of the RTX 5090 residency page's int8 note: symmetric, per row; on a
 * bandwidth-bound path halving the bytes halves the time). Each (position,
 * KV head) row of K and of V is stored as 128 int8 codes and one float scale:
 *   s = amax_r |x_r| / 127,  code_r = round_half_even(x_r / s)  (binary32,
 *   correctly rounded division; an all-zero row has s = 0),
 * and read back as code * s. K is quantized after RoPE and its bf16 rounding,
 * V as written. A row costs 2 x 128 + 8 bytes instead of 512.
 *
 *   k_cache8, v_cache8  int8 [num_pages][Hkv][page_size][D] (layout as the
 *                       bf16 cache), 16-byte aligned
 *   k_scale, v_scale    float [num_pages][Hkv][page_size], 16-byte aligned
 *
 * qk_norm_rope_append_int8 -- qk_norm_rope_append writing the new token's K
 *   and V rows into the INT8 cache (codes and scales); q_out as before.
 * decode_attn_paged_int8 -- decode_attn_paged over the INT8 cache: the same
 *   attention with every key and value row dequantized. The query must lie
 *   in the fp16 range (|q| < 65504; the fold runs fp16 tensor-core MMAs).
 *   Reading and PDL rules as decode_attn_paged; workspace of
 *   decode_attn_int8_workspace_size bytes with decode_attn_paged's rules
 *   (zero-filled before the first call with given arguments, left ready by
 *   every completed call, not shared by calls that may overlap); up to 64
 *   partitions whose states fit the CTA's shared memory are merged by the
 *   last CTA of each (sequence, KV head), more by a merge kernel in the same
 *   stream. The CTA shape follows the sizes as for decode_attn_paged (one,
 *   two or four CTAs per SM), so results are reproducible per device.
 */
int qk_norm_rope_append_int8(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                             const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                             const int32_t *context_lens, const int32_t *block_table, int8_t *k_cache8,
                             int8_t *v_cache8, float *k_scale, float *v_scale, pgqa_bf16 *q_out, int B,
                             int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                             float rope_theta, float eps, cudaStream_t stream);
size_t decode_attn_int8_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                       int num_partitions);
int decode_attn_paged_int8(const pgqa_bf16 *q, const int8_t *k_cache8, const int8_t *v_cache8,
                           const float *k_scale, const float *v_scale, const int32_t *block_table,
                           const int32_t *context_lens, int B, int Hq, int Hkv, int D, int page_size,
                           int max_pages, int num_pages, float scale, int num_partitions, float *out_f32,
                           pgqa_bf16 *out_bf16, void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * decode_step_paged_int8 -- qk_norm_rope_append_int8 followed by
 * decode_attn_paged_int8 in one launch, with the same results as calling the
 * two in order (as decode_step_paged is for the bf16 cache). Each attention
 * CTA normalises and rotates the query heads it serves; the CTA whose
 * partition holds position T_b - 1 quantizes the new K and V rows and writes
 * their codes and scales to the cache.
 *
 *   q, k, v, gamma_q, gamma_k, context_lens (T_b >= 1), block_table,
 *   k_cache8, v_cache8, k_scale, v_scale, rope_theta, eps
 *                                   as for qk_norm_rope_append_int8
 *   q_out    [B][Hq][D] bf16, nullable: the rotated query, if wanted
 *   scale, num_partitions, out_f32, out_bf16, workspace, ws_bytes
 *                                   as for decode_attn_paged_int8
 * Sequences with T_b < 1 raise PGQA_DEVERR_BAD_CONTEXT and produce zeros.
 */
int decode_step_paged_int8(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                           const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k, const int32_t *context_lens,
                           const int32_t *block_table, int8_t *k_cache8, int8_t *v_cache8, float *k_scale,
                           float *v_scale, pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D, int page_size,
                           int max_pages, int num_pages, float rope_theta, float eps, float scale,
                           int num_partitions, float *out_f32, pgqa_bf16 *out_bf16, void *workspace,
                           size_t ws_bytes, cudaStream_t stream);

/*
 * attn_partition_merge -- exact merge of NP partition states (s9.1).
 *   m, l  [B][Hq][NP] float   running max of the scores (natural-log units)
 *                             and the softmax denominator, both relative to m
 *   acc   [B][Hq][NP][D]      unnormalised weighted sums of V relative to m
 *   out = sum_p acc_p e^(m_p - M) / sum_p l_p e^(m_p - M), M = max_p m_p;
 *   zeros when the denominator is 0. Empty partitions (m = -1e30, l = 0,
 *   acc = 0) contribute nothing. 1 <= NP <= 65536.
 */
int attn_partition_merge(const float *m, const float *l, const float *acc, int B, int Hq, int D,
                         int NP, float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream);

/*
 * Host-tiled variant ("EdgeTransformerEngine", KV-offload design): the
 * state (m, l, acc) lives in global memory across KV tiles, so device memory
 * for KV is constant in the context length.
 *   m, l  [B][Hq] float, acc [B][Hq][D] float (natural-log units as above).
 *
 * attn_tile_init     m = -1e30, l = 0, acc = 0.
 * attn_tile_update   fold one tile of n_pos (1..512) consecutive positions
 *                    into the state with the online-softmax update:
 *                    k_tile, v_tile [B][n_pos][Hkv][D] bf16, q [B][Hq][D] bf16.
 * attn_tile_finalize out = acc / l (zeros where l = 0).
 */
int attn_tile_init(float *m, float *l, float *acc, int B, int Hq, int D, cudaStream_t stream);
int attn_tile_update(const pgqa_bf16 *q, const pgqa_bf16 *k_tile, const pgqa_bf16 *v_tile,
                     int n_pos, int B, int Hq, int Hkv, int D, float scale, float *m, float *l,
                     float *acc, cudaStream_t stream);
int attn_tile_finalize(const float *m, const float *l, const float *acc, int B, int Hq, int D,
                       float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream);

/*
 * attn_host_tiled_run -- enqueue the whole host-tiled attention: init, then
 * for each group g of tiles_per_copy consecutive tiles of tile_len positions
 * (the last group and tile may be shorter) one copy of K and one of V from
 * pinned host memory into device slot s = g % n_slots on copy_stream, then
 * attn_tile_update for each of the group's tiles in order on
 * compute_stream, then finalize. Two event dependencies per slot order the
 * slots (copy_done[s]: data ready before it is read; compute_done[s]: slot
 * free before it is overwritten), so copies of later tiles overlap the
 * updates of earlier ones. tiles_per_copy = 1 is the one-tile-per-copy
 * pipeline of [EdgeTransformerEngine]'s KV-offload design; larger groups
 * keep its 512-position tile updates and state but move the data in fewer,
 * larger copies, which the host link serves faster.
 *
 *   host_k, host_v  [B][T][Hkv][D] bf16, pinned host memory
 *   k_slots, v_slots  host arrays of n_slots device pointers, each slot
 *                     [B][tiles_per_copy * tile_len][Hkv][D] bf16;
 *                     2 <= n_slots <= 8
 *   events          host array of 2 * n_slots caller-created events
 *                   (copy_done[0..n_slots), then compute_done[0..n_slots))
 *   tile_len        1..512;  tiles_per_copy  1..64
 * Returns after enqueueing; the output is ready when compute_stream reaches
 * the end of the enqueued work. The streams must differ.
 */
int attn_host_tiled_run(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v,
                        int T, int B, int Hq, int Hkv, int D, float scale, int tile_len,
                        int tiles_per_copy, int n_slots, pgqa_bf16 *const *k_slots,
                        pgqa_bf16 *const *v_slots, cudaEvent_t const *events, float *m, float *l,
                        float *acc, float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t compute_stream,
                        cudaStream_t copy_stream);

/*
 * attn_host_tiled_run_traced -- attn_host_tiled_run that also records
 * caller-created events around every copy and every group of tile updates,
 * so that the overlap of copies and updates can be measured ("EdgeTransformer
 * Engine", KV-offload design and its current-limits list: the overlap there
 * was inferred, not measured). Same arguments and results, plus:
 *   trace_events    4 * n_trace_groups events created by the caller with
 *                   timing enabled; for copy group g < n_trace_groups (the
 *                   g-th copy of tiles_per_copy tiles):
 *                     [4g]     before the group's K copy   (copy_stream)
 *                     [4g + 1] after its V copy            (copy_stream)
 *                     [4g + 2] before its first tile update (compute_stream,
 *                              after the wait for the copy)
 *                     [4g + 3] after its last tile update  (compute_stream)
 *                   Groups past n_trace_groups are not traced.
 * PGQA_ERR_INVALID_ARG for a NULL event or a negative count. Nothing is
 * allocated.
 */
int attn_host_tiled_run_traced(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v, int T,
                               int B, int Hq, int Hkv, int D, float scale, int tile_len, int tiles_per_copy,
                               int n_slots, pgqa_bf16 *const *k_slots, pgqa_bf16 *const *v_slots,
                               cudaEvent_t const *events, float *m, float *l, float *acc, float *out_f32,
                               pgqa_bf16 *out_bf16, cudaStream_t compute_stream, cudaStream_t copy_stream,
                               cudaEvent_t const *trace_events, int n_trace_groups);

/*
 * Zero-copy variant of the host-tiled attention ([EdgeTransformerEngine],
 * KV-offload design, whose state (m, l, acc) and exact merge it keeps): the
 * history stays in pinned host memory and the kernel reads it over the host
 * link directly, with no device tiles and no copies. The history is split
 * into num_partitions ranges of consecutive positions, one CTA per (range, KV
 * head, sequence); their states are merged exactly as in
 * attn_partition_merge.
 *
 *   q            [B][Hq][D] bf16, device memory
 *   host_k, host_v  [B][T][Hkv][D] bf16, pinned host memory mapped into the
 *                device address space (cudaHostAlloc, or cudaHostRegister
 *                with mapping); PGQA_ERR_INVALID_ARG if it is not. The caller
 *                keeps it alive and unmodified until the stream passes the
 *                call.
 *   num_partitions  0 = automatic (one wave of CTAs, ranges >= 512
 *                positions), else the requested count (clamped to [1, T]).
 *   workspace    device scratch of ws_bytes >= attn_host_direct_workspace_size
 *                (may be NULL when that size is 0); no initial value needed.
 *   out_f32, out_bf16  [B][Hq][D], at least one non-NULL.
 * T = 0 produces zeros. Reads q after the previous kernel in the stream
 * completes (programmatic stream serialisation).
 */
int attn_host_direct_partition_count(int B, int Hkv, int T, int num_partitions);
size_t attn_host_direct_workspace_size(int B, int Hq, int Hkv, int T, int num_partitions);
int attn_host_direct(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v, int T,
                     int B, int Hq, int Hkv, int D, float scale, int num_partitions, float *out_f32,
                     pgqa_bf16 *out_bf16, void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * decode_attn_paged_static -- decode_attn_paged for callers that cannot
 * allocate device memory. The pages have no counterpart of this entry point;
 * it exists for code that runs where cudaMalloc is not allowed (inside an
 * allocator or memory-pool callback, in a plugin whose host owns all device
 * memory, in a loop that forbids allocation after start-up) and so cannot
 * provide decode_attn_paged's workspace.
 *
 * Same arguments and results as decode_attn_paged, without the workspace:
 * the partition scratch is a fixed array of PGQA_STATIC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the
 * process exits. Sizes whose scratch (decode_attn_workspace_size) exceeds it
 * are refused with PGQA_ERR_WORKSPACE and a message naming both sizes.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *
 * The first call on each device (that needs scratch) looks the array's
 * device address up with cudaGetSymbolAddress and keeps it with the id of
 * the device's current context; the first call after that context is torn
 * down and made again (cudaDeviceReset) looks it up again. Make the first
 * call on a device, and the first after a reset, before any stream capture
 * on that device. All calls share the one array, which
 * keeps the last call's contents: each call first clears the part that must
 * start at zero (the partition tickets) with cudaMemsetAsync on `stream`.
 * Calls whose work overlaps on the GPU (different streams, or no ordering
 * between them) race on the array and must not be issued.
 */
#define PGQA_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

int decode_attn_paged_static(const pgqa_bf16 *q, const pgqa_bf16 *k_cache,
                             const pgqa_bf16 *v_cache, const int32_t *block_table,
                             const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                             int page_size, int max_pages, int num_pages, float scale,
                             int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PGQA_H */
