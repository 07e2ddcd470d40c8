/*
 * oracle.c -- plain, slow, fp64 CPU statement of the single-token paged GQA
 * decode step.
 *
 * TEST INFRASTRUCTURE. This file is the oracle that the CUDA library is
 * checked against. Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table
 * or helper with the CUDA library, and the CUDA library never includes, links
 * or calls it.
 *
 * Everything is computed in double precision. The attention routine writes
 * out every score and the full softmax; there is no blocking, fusion or
 * reordering beyond what the definitions state. Inputs are the same bf16 bit
 * patterns the GPU receives (uint16_t), widened exactly to double.
 *
 * Sources (page title, then the section on that page):
 *   [EdgeTransformerEngine]  "EdgeTransformerEngine" (thomasli.cn, cuda-engine):
 *       online-softmax note (state (m, l, acc) and its update step),
 *       KV-offload design (attn_init / attn_tile / attn_finalize, m = -1e30),
 *       bf16-as-storage note (bf16 is the top half of a binary32).
 *   [Qwen3 runtime]  "From Qwen3 math to CUDA kernels: a 0.6B inference
 *       runtime" (chengzipai.xyz):
 *       s0.1 precision roles, s2.1 RMSNorm (eps = 1e-6), s2.3 Q/K head
 *       RMSNorm, s2.4 RoPE as a 2-D rotation of the pair (i, i + D/2),
 *       s2.5 GQA head map, s2.6 scaled dot-product attention with the causal
 *       mask j <= t, s7.2 logical token -> physical cache address,
 *       s9.1 exact merge of partitions.
 *
 * Readings where those pages are silent (their formulas were lost in text
 * extraction) are stated beside each function.
 *
 * Parity pins: every function below is pinned by a test under tests/ that
 * does not restate its formula (closed forms, invariants, special cases,
 * agreement of two different algorithms, a library rounding routine).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes of the oracle's entry points. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEMORY (-2)

/* ------------------------------------------------------------------------- */
/* bf16 storage [EdgeTransformerEngine, bf16-as-storage note;                */
/*               Qwen3 runtime s0.1]                                          */
/* ------------------------------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening puts the
 * 16 bits on top and zero-fills the rest, which is exact. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (8 significant bits,
 * binary32 exponent range, gradual underflow, overflow to infinity).
 * Reading: bf16 I/O with round-to-nearest-even is the only rounding the pages
 * name for storing results (Qwen3 runtime s0.1: results go back to bf16). */
uint16_t oracle_round_bf16(double x)
{
    if (isnan(x))
        return (uint16_t)0x7FC0u;
    uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    /* Largest finite bf16 is (2 - 2^-7) * 2^127; the midpoint to 2^128 rounds
     * to the even neighbour, which is infinity. */
    const double overflow_mid = ldexp(2.0 - ldexp(1.0, -8), 127);
    if (a >= overflow_mid)
        return (uint16_t)(sign | 0x7F80u);
    int e2; /* a = f * 2^e2, f in [0.5, 1): leading bit has weight 2^(e2-1) */
    (void)frexp(a, &e2);
    int lead = e2 - 1;
    if (lead < -126)
        lead = -126; /* subnormal range: fixed quantum 2^-133 */
    double quantum = ldexp(1.0, lead - 7);
    double r = rint(a / quantum) * quantum; /* rint rounds half to even */
    float rf = (float)r;                    /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* ------------------------------------------------------------------------- */
/* A3: per-head RMSNorm [Qwen3 runtime s2.1 definition, s2.3 per head]       */
/* ------------------------------------------------------------------------- */

/* out_r = x_r * gamma_r / sqrt(mean_r(x_r^2) + eps), over one head of D
 * values. Reading: s2.3's formula was lost; it reuses s2.1's RMSNorm on the
 * head vector, gamma has one weight per in-head dimension r. */
void oracle_head_rmsnorm(const double *x, const double *gamma, int D, double eps,
                         double *out)
{
    double sum_sq = 0.0;
    for (int r = 0; r < D; ++r)
        sum_sq += x[r] * x[r];
    double inv_rms = 1.0 / sqrt(sum_sq / (double)D + eps);
    for (int r = 0; r < D; ++r)
        out[r] = x[r] * inv_rms * gamma[r];
}

/* ------------------------------------------------------------------------- */
/* A4: half-rotation RoPE [Qwen3 runtime s2.4; s7.1 pairs (r, r+64)]         */
/* ------------------------------------------------------------------------- */

/* For i < D/2: omega_i = theta^(-2i/D), phi = pos * omega_i,
 * (a, b) = (x_i, x_{i+D/2}) -> (a cos phi - b sin phi, b cos phi + a sin phi).
 * Reading: s2.4 names the angular frequency, the phase and the pairing of the
 * two halves; the formulas themselves were lost, so the standard rotary form
 * with a counter-clockwise rotation is taken. */
void oracle_rope_half(const double *x, int D, long pos, double theta, double *out)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double omega = pow(theta, -2.0 * (double)i / (double)D);
        double phi = (double)pos * omega;
        double c = cos(phi), s = sin(phi);
        double a = x[i], b = x[i + half];
        out[i] = a * c - b * s;
        out[i + half] = b * c + a * s;
    }
}

/* ------------------------------------------------------------------------- */
/* A5: GQA head map [Qwen3 runtime s2.5]                                     */
/* ------------------------------------------------------------------------- */

/* Query head h reads KV head h / (Hq / Hkv) (integer division). */
int oracle_kv_head(int h, int Hq, int Hkv) { return h / (Hq / Hkv); }

/* ------------------------------------------------------------------------- */
/* A7: paged addressing [Qwen3 runtime s7.2]                                  */
/* ------------------------------------------------------------------------- */

/* Element offset of the D-vector of (sequence b, KV head kvh, position pos)
 * in a cache laid out [num_pages][Hkv][P][D]:
 *   logical page l = pos / P, in-page offset o = pos % P,
 *   physical page q = block_table[b][l],
 *   offset = ((q * Hkv + kvh) * P + o) * D.
 * Returns -1 when the table entry lies outside [0, num_pages).
 * Reading: s7.2 gives l, o and q; the layout inside a page is not given, so
 * [Hkv][P][D] per page is this library's choice. */
long oracle_cache_offset(const int32_t *block_table, int max_pages, int num_pages, int b,
                         int kvh, long pos, int Hkv, int P, int D)
{
    long logical = pos / P;
    long in_page = pos % P;
    if (logical < 0 || logical >= max_pages)
        return -1;
    int32_t phys = block_table[(long)b * max_pages + logical];
    if (phys < 0 || phys >= num_pages)
        return -1;
    return (((long)phys * Hkv + kvh) * P + in_page) * (long)D;
}

/* ------------------------------------------------------------------------- */
/* Prologue: A3 + A4 + append [Qwen3 runtime s2.3, s2.4, s7.1, s7.2]          */
/* ------------------------------------------------------------------------- */

/* For every sequence b with context length T = context_lens[b] (T counts the
 * new token), the new token sits at pos = T - 1:
 *   q_out[b][h]  = bf16(RoPE_pos(RMSNorm(q[b][h], gamma_q)))      h < Hq
 *   K slot       = bf16(RoPE_pos(RMSNorm(k[b][h], gamma_k)))      h < Hkv
 *   V slot       = v[b][h] (bit copy, V gets no norm)              h < Hkv
 * The K and V slots are the (b, h, pos) rows of k_cache / v_cache; nothing
 * else in either cache is written.
 * Readings: norm then RoPE (the order of the page's per-layer chain); the new
 * token's position is T - 1. Returns ORACLE_BAD_ARG for T < 1, T beyond the
 * block table, or a table entry outside the pool. */
int oracle_qk_norm_rope_append(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const uint16_t *gamma_q, const uint16_t *gamma_k,
                               const int32_t *context_lens, const int32_t *block_table,
                               uint16_t *k_cache, uint16_t *v_cache, uint16_t *q_out, int B,
                               int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                               double theta, double eps)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) != 0 || P <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    double *x = malloc(sizeof(double) * (size_t)D * 4);
    if (!x)
        return ORACLE_NO_MEMORY;
    double *gam = x + D, *nrm = x + 2 * D, *rot = x + 3 * D;
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        if (T < 1 || T > (long)max_pages * P) {
            status = ORACLE_BAD_ARG;
            break;
        }
        long pos = T - 1;
        for (int h = 0; h < Hq; ++h) {
            for (int r = 0; r < D; ++r) {
                x[r] = oracle_bf16_to_double(q[((long)b * Hq + h) * D + r]);
                gam[r] = oracle_bf16_to_double(gamma_q[r]);
            }
            oracle_head_rmsnorm(x, gam, D, eps, nrm);
            oracle_rope_half(nrm, D, pos, theta, rot);
            for (int r = 0; r < D; ++r)
                q_out[((long)b * Hq + h) * D + r] = oracle_round_bf16(rot[r]);
        }
        for (int h = 0; h < Hkv; ++h) {
            long off = oracle_cache_offset(block_table, max_pages, num_pages, b, h, pos, Hkv, P, D);
            if (off < 0) {
                status = ORACLE_BAD_ARG;
                break;
            }
            for (int r = 0; r < D; ++r) {
                x[r] = oracle_bf16_to_double(k[((long)b * Hkv + h) * D + r]);
                gam[r] = oracle_bf16_to_double(gamma_k[r]);
            }
            oracle_head_rmsnorm(x, gam, D, eps, nrm);
            oracle_rope_half(nrm, D, pos, theta, rot);
            for (int r = 0; r < D; ++r) {
                k_cache[off + r] = oracle_round_bf16(rot[r]);
                v_cache[off + r] = v[((long)b * Hkv + h) * D + r];
            }
        }
    }
    free(x);
    return status;
}

/* The prologue for M new tokens per sequence: token i of sequence b (q row
 * [b][i][h], k and v rows [b][i][h]) sits at position T - M + i and gets the
 * same treatment as the single new token of oracle_qk_norm_rope_append at
 * that position (q_out [B][M][Hq][D]; K slot rotated, V slot copied).
 * Returns ORACLE_BAD_ARG for T < M or an unusable slot. */
int oracle_qk_norm_rope_append_multi(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const uint16_t *gamma_q, const uint16_t *gamma_k,
                                     const int32_t *context_lens, const int32_t *block_table,
                                     uint16_t *k_cache, uint16_t *v_cache, uint16_t *q_out, int B,
                                     int M, int Hq, int Hkv, int D, int P, int max_pages,
                                     int num_pages, double theta, double eps)
{
    if (B < 0 || M < 1 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) != 0 || P <= 0 ||
        Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    double *x = malloc(sizeof(double) * (size_t)D * 4);
    if (!x)
        return ORACLE_NO_MEMORY;
    double *gam = x + D, *nrm = x + 2 * D, *rot = x + 3 * D;
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        if (T < M || T > (long)max_pages * P) {
            status = ORACLE_BAD_ARG;
            break;
        }
        for (int i = 0; i < M && status == ORACLE_OK; ++i) {
            long pos = T - M + i;
            long tok = (long)b * M + i;
            for (int h = 0; h < Hq; ++h) {
                for (int r = 0; r < D; ++r) {
                    x[r] = oracle_bf16_to_double(q[(tok * Hq + h) * D + r]);
                    gam[r] = oracle_bf16_to_double(gamma_q[r]);
                }
                oracle_head_rmsnorm(x, gam, D, eps, nrm);
                oracle_rope_half(nrm, D, pos, theta, rot);
                for (int r = 0; r < D; ++r)
                    q_out[(tok * Hq + h) * D + r] = oracle_round_bf16(rot[r]);
            }
            for (int h = 0; h < Hkv; ++h) {
                long off = oracle_cache_offset(block_table, max_pages, num_pages, b, h, pos, Hkv, P,
                                               D);
                if (off < 0) {
                    status = ORACLE_BAD_ARG;
                    break;
                }
                for (int r = 0; r < D; ++r) {
                    x[r] = oracle_bf16_to_double(k[(tok * Hkv + h) * D + r]);
                    gam[r] = oracle_bf16_to_double(gamma_k[r]);
                }
                oracle_head_rmsnorm(x, gam, D, eps, nrm);
                oracle_rope_half(nrm, D, pos, theta, rot);
                for (int r = 0; r < D; ++r) {
                    k_cache[off + r] = oracle_round_bf16(rot[r]);
                    v_cache[off + r] = v[(tok * Hkv + h) * D + r];
                }
            }
        }
    }
    free(x);
    return status;
}

/* ------------------------------------------------------------------------- */
/* INT8 KV rows [Qwen3 runtime s0.1: INT8 values times an FP32 scale,        */
/*   accumulated in FP32; RTX 5090 residency page: int8 symmetric per-row     */
/*   quantization halves the bytes a bandwidth-bound path moves]              */
/* ------------------------------------------------------------------------- */

/* Symmetric per-row quantization of one D-vector given as bf16 bits (a K row
 * after RoPE and its bf16 rounding, or a V row as written):
 *   amax = max_r |x_r|,  s = amax / 127,  code_r = round_half_even(x_r / s)
 * (codes in [-127, 127]; an all-zero row has s = 0 and zero codes).
 * Reading: the pages fix int8, symmetric, per row and an FP32 scale; the row
 * here is one (position, KV head) vector. The scale and the quotients are
 * formed in binary32 -- the precision in which the kernel takes the same
 * integer decision -- with correctly rounded division. */
void oracle_quantize_row_int8(const uint16_t *row, int D, int8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int r = 0; r < D; ++r) {
        float a = fabsf((float)oracle_bf16_to_double(row[r]));
        if (a > amax)
            amax = a;
    }
    volatile float s = amax / 127.0f; /* binary32, rounded once */
    *scale = s;
    for (int r = 0; r < D; ++r) {
        if (amax == 0.0f) {
            codes[r] = 0;
            continue;
        }
        volatile float quot = (float)oracle_bf16_to_double(row[r]) / s;
        float c = rintf(quot); /* round half to even (default rounding mode) */
        if (c > 127.0f)
            c = 127.0f;
        if (c < -127.0f)
            c = -127.0f;
        codes[r] = (int8_t)c;
    }
}

/* oracle_quantize_row_int8 applied to n consecutive rows of D values
 * (a whole cache [num_pages][Hkv][P][D] -> codes of the same shape and one
 * scale per row). */
void oracle_quantize_rows_int8(const uint16_t *rows, long n, int D, int8_t *codes, float *scales)
{
    for (long i = 0; i < n; ++i)
        oracle_quantize_row_int8(rows + i * D, D, codes + i * D, scales + i);
}

/* Dequantized value code * scale, exact in double. */
double oracle_dequant_int8(int8_t code, float scale) { return (double)code * (double)scale; }

/* The prologue with an INT8 cache: as oracle_qk_norm_rope_append, except that
 * the K slot receives the int8 codes and the scale of the bf16-rounded
 * rotated K row, and the V slot those of the V row. Caches are int8
 * [num_pages][Hkv][P][D], scales float [num_pages][Hkv][P]. */
int oracle_qk_norm_rope_append_int8(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                    const uint16_t *gamma_q, const uint16_t *gamma_k,
                                    const int32_t *context_lens, const int32_t *block_table,
                                    int8_t *k_cache, int8_t *v_cache, float *k_scale,
                                    float *v_scale, uint16_t *q_out, int B, int Hq, int Hkv, int D,
                                    int P, int max_pages, int num_pages, double theta, double eps)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) != 0 || P <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    double *x = malloc(sizeof(double) * (size_t)D * 4);
    uint16_t *kb = malloc(sizeof(uint16_t) * (size_t)D);
    if (!x || !kb) {
        free(x), free(kb);
        return ORACLE_NO_MEMORY;
    }
    double *gam = x + D, *nrm = x + 2 * D, *rot = x + 3 * D;
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        if (T < 1 || T > (long)max_pages * P) {
            status = ORACLE_BAD_ARG;
            break;
        }
        long pos = T - 1;
        for (int h = 0; h < Hq; ++h) {
            for (int r = 0; r < D; ++r) {
                x[r] = oracle_bf16_to_double(q[((long)b * Hq + h) * D + r]);
                gam[r] = oracle_bf16_to_double(gamma_q[r]);
            }
            oracle_head_rmsnorm(x, gam, D, eps, nrm);
            oracle_rope_half(nrm, D, pos, theta, rot);
            for (int r = 0; r < D; ++r)
                q_out[((long)b * Hq + h) * D + r] = oracle_round_bf16(rot[r]);
        }
        for (int h = 0; h < Hkv; ++h) {
            long off = oracle_cache_offset(block_table, max_pages, num_pages, b, h, pos, Hkv, P, D);
            if (off < 0) {
                status = ORACLE_BAD_ARG;
                break;
            }
            for (int r = 0; r < D; ++r) {
                x[r] = oracle_bf16_to_double(k[((long)b * Hkv + h) * D + r]);
                gam[r] = oracle_bf16_to_double(gamma_k[r]);
            }
            oracle_head_rmsnorm(x, gam, D, eps, nrm);
            oracle_rope_half(nrm, D, pos, theta, rot);
            for (int r = 0; r < D; ++r)
                kb[r] = oracle_round_bf16(rot[r]);
            long row = off / D; /* (page, head, slot) index of the scale arrays */
            oracle_quantize_row_int8(kb, D, k_cache + off, k_scale + row);
            oracle_quantize_row_int8(v + ((long)b * Hkv + h) * D, D, v_cache + off, v_scale + row);
        }
    }
    free(x), free(kb);
    return status;
}

/* ------------------------------------------------------------------------- */
/* A5 + A6: decode attention, full softmax [Qwen3 runtime s2.5, s2.6]        */
/* ------------------------------------------------------------------------- */

/* One query head against T gathered keys/values (row j of keys/values is the
 * D-vector at position j):
 *   s_j = scale * sum_r q_r K_jr                 for j = 0 .. T-1 (causal j <= t)
 *   w_j = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
 *   out_r = sum_j w_j V_jr
 * T = 0 gives zeros. The full score vector and softmax are materialised. */
static void softmax_attend(const double *qv, const double *keys, const double *values, long T,
                           int D, double scale, double *scores, double *out)
{
    for (int r = 0; r < D; ++r)
        out[r] = 0.0;
    if (T <= 0)
        return;
    double smax = -INFINITY;
    for (long j = 0; j < T; ++j) {
        double dot = 0.0;
        for (int r = 0; r < D; ++r)
            dot += qv[r] * keys[j * D + r];
        scores[j] = scale * dot;
        if (scores[j] > smax)
            smax = scores[j];
    }
    double z = 0.0;
    for (long j = 0; j < T; ++j) {
        scores[j] = exp(scores[j] - smax);
        z += scores[j];
    }
    for (long j = 0; j < T; ++j) {
        double w = scores[j] / z;
        for (int r = 0; r < D; ++r)
            out[r] += w * values[j * D + r];
    }
}

/* Decode attention over the paged cache. For each sequence b (context length
 * T = context_lens[b]) and query head h < Hq, gather the T keys and values
 * of KV head h / (Hq/Hkv) position by position through the block table, then
 * apply softmax_attend. out is double [B][Hq][D].
 * Reading: scale is a parameter (1/sqrt(D) in every workload here). */
int oracle_decode_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_table, const int32_t *context_lens, int B,
                            int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                            double scale, double *out)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    long Tmax = 0;
    for (int b = 0; b < B; ++b) {
        if (context_lens[b] < 0 || (long)context_lens[b] > (long)max_pages * P)
            return ORACLE_BAD_ARG;
        if (context_lens[b] > Tmax)
            Tmax = context_lens[b];
    }
    size_t n = (size_t)(Tmax > 0 ? Tmax : 1);
    double *keys = malloc(sizeof(double) * n * (size_t)D);
    double *values = malloc(sizeof(double) * n * (size_t)D);
    double *scores = malloc(sizeof(double) * n);
    double *qv = malloc(sizeof(double) * (size_t)D);
    if (!keys || !values || !scores || !qv) {
        free(keys), free(values), free(scores), free(qv);
        return ORACLE_NO_MEMORY;
    }
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        for (int h = 0; h < Hq && status == ORACLE_OK; ++h) {
            int kvh = oracle_kv_head(h, Hq, Hkv);
            for (long j = 0; j < T; ++j) {
                long off = oracle_cache_offset(block_table, max_pages, num_pages, b, kvh, j, Hkv,
                                               P, D);
                if (off < 0) {
                    status = ORACLE_BAD_ARG;
                    break;
                }
                for (int r = 0; r < D; ++r) {
                    keys[j * D + r] = oracle_bf16_to_double(k_cache[off + r]);
                    values[j * D + r] = oracle_bf16_to_double(v_cache[off + r]);
                }
            }
            if (status != ORACLE_OK)
                break;
            for (int r = 0; r < D; ++r)
                qv[r] = oracle_bf16_to_double(q[((long)b * Hq + h) * D + r]);
            softmax_attend(qv, keys, values, T, D, scale, scores, out + ((long)b * Hq + h) * D);
        }
    }
    free(keys), free(values), free(scores), free(qv);
    return status;
}

/* Multi-query decode: M new tokens per sequence. With T = context_lens[b]
 * (counting all M new tokens), token i (0 <= i < M) sits at position
 * t_i = T - M + i and, being causal (j <= t_i), attends to positions
 * 0 .. t_i, i.e. to the first T - M + i + 1 keys: for each (b, i, h),
 * softmax_attend over those keys of KV head h / (Hq/Hkv). q and out are
 * [B][M][Hq][D]. Returns ORACLE_BAD_ARG for T < M. */
int oracle_decode_attention_multi(const uint16_t *q, const uint16_t *k_cache,
                                  const uint16_t *v_cache, const int32_t *block_table,
                                  const int32_t *context_lens, int B, int M, int Hq, int Hkv,
                                  int D, int P, int max_pages, int num_pages, double scale,
                                  double *out)
{
    if (B < 0 || M < 1 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    long Tmax = 0;
    for (int b = 0; b < B; ++b) {
        if (context_lens[b] < M || (long)context_lens[b] > (long)max_pages * P)
            return ORACLE_BAD_ARG;
        if (context_lens[b] > Tmax)
            Tmax = context_lens[b];
    }
    size_t n = (size_t)(Tmax > 0 ? Tmax : 1);
    double *keys = malloc(sizeof(double) * n * (size_t)D);
    double *values = malloc(sizeof(double) * n * (size_t)D);
    double *scores = malloc(sizeof(double) * n);
    double *qv = malloc(sizeof(double) * (size_t)D);
    if (!keys || !values || !scores || !qv) {
        free(keys), free(values), free(scores), free(qv);
        return ORACLE_NO_MEMORY;
    }
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        for (int h = 0; h < Hq && status == ORACLE_OK; ++h) {
            int kvh = oracle_kv_head(h, Hq, Hkv);
            for (long j = 0; j < T; ++j) {
                long off = oracle_cache_offset(block_table, max_pages, num_pages, b, kvh, j, Hkv,
                                               P, D);
                if (off < 0) {
                    status = ORACLE_BAD_ARG;
                    break;
                }
                for (int r = 0; r < D; ++r) {
                    keys[j * D + r] = oracle_bf16_to_double(k_cache[off + r]);
                    values[j * D + r] = oracle_bf16_to_double(v_cache[off + r]);
                }
            }
            if (status != ORACLE_OK)
                break;
            for (int i = 0; i < M; ++i) {
                long row = ((long)b * M + i) * Hq + h;
                for (int r = 0; r < D; ++r)
                    qv[r] = oracle_bf16_to_double(q[row * D + r]);
                long visible = T - M + i + 1; /* positions 0 .. t_i */
                softmax_attend(qv, keys, values, visible, D, scale, scores, out + row * D);
            }
        }
    }
    free(keys), free(values), free(scores), free(qv);
    return status;
}

/* Decode attention over an INT8 cache: oracle_decode_attention with every
 * key and value row replaced by its dequantized values code * scale. */
int oracle_decode_attention_int8(const uint16_t *q, const int8_t *k_cache, const int8_t *v_cache,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *block_table, const int32_t *context_lens, int B,
                                 int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                                 double scale, double *out)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    long Tmax = 0;
    for (int b = 0; b < B; ++b) {
        if (context_lens[b] < 0 || (long)context_lens[b] > (long)max_pages * P)
            return ORACLE_BAD_ARG;
        if (context_lens[b] > Tmax)
            Tmax = context_lens[b];
    }
    size_t n = (size_t)(Tmax > 0 ? Tmax : 1);
    double *keys = malloc(sizeof(double) * n * (size_t)D);
    double *values = malloc(sizeof(double) * n * (size_t)D);
    double *scores = malloc(sizeof(double) * n);
    double *qv = malloc(sizeof(double) * (size_t)D);
    if (!keys || !values || !scores || !qv) {
        free(keys), free(values), free(scores), free(qv);
        return ORACLE_NO_MEMORY;
    }
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        long T = context_lens[b];
        for (int h = 0; h < Hq && status == ORACLE_OK; ++h) {
            int kvh = oracle_kv_head(h, Hq, Hkv);
            for (long j = 0; j < T; ++j) {
                long off = oracle_cache_offset(block_table, max_pages, num_pages, b, kvh, j, Hkv,
                                               P, D);
                if (off < 0) {
                    status = ORACLE_BAD_ARG;
                    break;
                }
                long row = off / D;
                for (int r = 0; r < D; ++r) {
                    keys[j * D + r] = oracle_dequant_int8(k_cache[off + r], k_scale[row]);
                    values[j * D + r] = oracle_dequant_int8(v_cache[off + r], v_scale[row]);
                }
            }
            if (status != ORACLE_OK)
                break;
            for (int r = 0; r < D; ++r)
                qv[r] = oracle_bf16_to_double(q[((long)b * Hq + h) * D + r]);
            softmax_attend(qv, keys, values, T, D, scale, scores, out + ((long)b * Hq + h) * D);
        }
    }
    free(keys), free(values), free(scores), free(qv);
    return status;
}

/* Decode attention over an unpaged history laid out [B][T][Hkv][D] (the
 * layout of the host-resident K/V of the host-tiled variant). Same
 * definition as oracle_decode_attention with every sequence of length T. */
int oracle_attention_contiguous(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B,
                                long T, int Hq, int Hkv, int D, double scale, double *out)
{
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    size_t n = (size_t)(T > 0 ? T : 1);
    double *keys = malloc(sizeof(double) * n * (size_t)D);
    double *values = malloc(sizeof(double) * n * (size_t)D);
    double *scores = malloc(sizeof(double) * n);
    double *qv = malloc(sizeof(double) * (size_t)D);
    if (!keys || !values || !scores || !qv) {
        free(keys), free(values), free(scores), free(qv);
        return ORACLE_NO_MEMORY;
    }
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            int kvh = oracle_kv_head(h, Hq, Hkv);
            for (long j = 0; j < T; ++j) {
                long off = (((long)b * T + j) * Hkv + kvh) * (long)D;
                for (int r = 0; r < D; ++r) {
                    keys[j * D + r] = oracle_bf16_to_double(k[off + r]);
                    values[j * D + r] = oracle_bf16_to_double(v[off + r]);
                }
            }
            for (int r = 0; r < D; ++r)
                qv[r] = oracle_bf16_to_double(q[((long)b * Hq + h) * D + r]);
            softmax_attend(qv, keys, values, T, D, scale, scores, out + ((long)b * Hq + h) * D);
        }
    }
    free(keys), free(values), free(scores), free(qv);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* A1: online softmax state [EdgeTransformerEngine, online-softmax note;      */
/*     Qwen3 runtime s9.1 update_online_state]                               */
/* ------------------------------------------------------------------------- */

/* Start state of the KV-offload design: m = -1e30, l = 0, acc = 0. */
void oracle_state_init(int D, double *m, double *l, double *acc)
{
    *m = -1e30;
    *l = 0.0;
    for (int r = 0; r < D; ++r)
        acc[r] = 0.0;
}

/* Fold keys j = 0 .. n-1 (scores s_j, value rows V_j) into the state one at a
 * time, in the page's order:
 *   newm = max(m, s); ecorr = exp(m - newm); p = exp(s - newm);
 *   l = l * ecorr + p; acc = acc * ecorr + p * V; m = newm. */
void oracle_state_update(const double *scores, const double *values, long n, int D, double *m,
                         double *l, double *acc)
{
    for (long j = 0; j < n; ++j) {
        double newm = scores[j] > *m ? scores[j] : *m;
        double ecorr = exp(*m - newm);
        double p = exp(scores[j] - newm);
        *l = *l * ecorr + p;
        for (int r = 0; r < D; ++r)
            acc[r] = acc[r] * ecorr + p * values[j * D + r];
        *m = newm;
    }
}

/* out = acc / l (the finalize kernel of the KV-offload design); l = 0, which
 * only an empty history produces, gives zeros. */
void oracle_state_finalize(double l, const double *acc, int D, double *out)
{
    for (int r = 0; r < D; ++r)
        out[r] = l > 0.0 ? acc[r] / l : 0.0;
}

/* ------------------------------------------------------------------------- */
/* A2: exact merge of partitions [Qwen3 runtime s9.1]                         */
/* ------------------------------------------------------------------------- */

/* Partition p holds (m_p, l_p, o_p) with o_p = acc_p (an unnormalised D-vector).
 *   M = max_p m_p;  L = sum_p l_p exp(m_p - M);  O = sum_p o_p exp(m_p - M);
 *   out = O / L (zeros when L = 0).
 * m, l are [NP]; acc is [NP][D]. Empty partitions (m = -1e30, l = 0, acc = 0)
 * add exactly nothing. Reading: s9.1's formulas were lost; this is the
 * rescale-to-common-maximum it describes in words. */
void oracle_merge_partitions(const double *m, const double *l, const double *acc, int NP, int D,
                             double *out)
{
    double M = -INFINITY;
    for (int p = 0; p < NP; ++p)
        if (m[p] > M)
            M = m[p];
    double L = 0.0;
    for (int r = 0; r < D; ++r)
        out[r] = 0.0;
    for (int p = 0; p < NP; ++p) {
        double w = exp(m[p] - M);
        L += l[p] * w;
        for (int r = 0; r < D; ++r)
            out[r] += acc[(long)p * D + r] * w;
    }
    for (int r = 0; r < D; ++r)
        out[r] = L > 0.0 ? out[r] / L : 0.0;
}
