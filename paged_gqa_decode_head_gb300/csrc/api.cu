// api.cu -- the C ABI of libpgqa (declared in include/pgqa.h): argument
// validation, partition choice and launch. Every entry point returns a status
// code and records a message for pgqa_last_error(); none throws, allocates or
// synchronises (except pgqa_device_error, which reads the device flags).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <atomic>

#include "launch.h"
#include "pgqa.h"

namespace pgqa {
constexpr int kHeadDimHost = 128;
constexpr int kMaxGroupHost = 8; // columns (query, head pairs) one decode CTA serves
}

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_last_error[0] = '\0';
    return PGQA_OK;
}

int cuda_fail(cudaError_t err, const char *where)
{
    return fail(PGQA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Shape checks common to every attention entry point. Returns 0 or a status.
int check_heads(const char *fn, int B, int Hq, int Hkv, int D)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: need B >= 0, Hq > 0, Hkv > 0 (got %d, %d, %d)", fn, B,
                    Hq, Hkv);
    if (B > 65535)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: B = %d exceeds 65535", fn, B);
    if (D != pgqa::kHeadDimHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: head dim %d unsupported (only 128)", fn, D);
    if (Hq % Hkv != 0)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: Hq = %d is not a multiple of Hkv = %d", fn, Hq, Hkv);
    const int g = Hq / Hkv;
    if (g < 1 || g > 8)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: group size Hq/Hkv = %d outside [1, 8]", fn, g);
    return 0;
}

int check_pages(const char *fn, int page_size, int max_pages, int num_pages)
{
    if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: page_size %d is not a power of two in [16, 256]", fn,
                    page_size);
    if (max_pages < 0 || num_pages < 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: negative max_pages or num_pages", fn);
    if (static_cast<long long>(max_pages) * page_size > 0x7FFFFFFFLL)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: max_pages * page_size exceeds 2^31 - 1", fn);
    return 0;
}

int sm_count_current_device()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

} // namespace

int pgqa::report_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

extern "C" {

const char *pgqa_last_error(void) { return g_last_error; }

int pgqa_device_error(unsigned *flags_out, int clear)
{
    if (!flags_out)
        return fail(PGQA_ERR_INVALID_ARG, "pgqa_device_error: flags_out is NULL");
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess)
        return cuda_fail(err, "pgqa_device_error");
    unsigned a = 0, b = 0, c = 0;
    if ((err = pgqa::read_flags_prologue(&a, clear != 0)) != cudaSuccess)
        return cuda_fail(err, "pgqa_device_error");
    if ((err = pgqa::read_flags_decode(&b, clear != 0)) != cudaSuccess)
        return cuda_fail(err, "pgqa_device_error");
    if ((err = pgqa::read_flags_int8(&c, clear != 0)) != cudaSuccess)
        return cuda_fail(err, "pgqa_device_error");
    *flags_out = a | b | c;
    return ok();
}

int pgqa_selftest_wait_timeout(cudaStream_t stream)
{
    cudaError_t err = pgqa::launch_wait_selftest(stream);
    if (err != cudaSuccess)
        return cuda_fail(err, "pgqa_selftest_wait_timeout");
    return ok();
}

static int prologue_impl(const char *fn, int M, const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                        const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                        const int32_t *context_lens, const int32_t *block_table,
                        pgqa_bf16 *k_cache, pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq,
                        int Hkv, int D, int page_size, int max_pages, int num_pages,
                        float rope_theta, float eps, cudaStream_t stream)
{
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (int st = check_pages(fn, page_size, max_pages, num_pages))
        return st;
    if (!(rope_theta > 0.f) || !std::isfinite(rope_theta) || !(eps >= 0.f) || !std::isfinite(eps))
        return fail(PGQA_ERR_INVALID_ARG, "%s: rope_theta must be > 0 and eps >= 0", fn);
    if (M < 1 || M > 64)
        return fail(PGQA_ERR_INVALID_ARG, "%s: M = %d new tokens per sequence outside [1, 64]", fn, M);
    if (B == 0)
        return ok();
    if (!q || !k || !v || !gamma_q || !gamma_k || !context_lens || !block_table || !k_cache ||
        !v_cache || !q_out)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gamma_q) ||
        !aligned16(gamma_k) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_out) ||
        !aligned4(context_lens) || !aligned4(block_table))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte and index arrays 4-byte alignment", fn);
    pgqa::PrologueArgs a{q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache,
                         q_out, B, Hq, Hkv, page_size, max_pages, num_pages,
                         static_cast<double>(rope_theta), eps, M};
    cudaError_t err = pgqa::launch_prologue(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int qk_norm_rope_append(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                        const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                        const int32_t *context_lens, const int32_t *block_table,
                        pgqa_bf16 *k_cache, pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq,
                        int Hkv, int D, int page_size, int max_pages, int num_pages,
                        float rope_theta, float eps, cudaStream_t stream)
{
    return prologue_impl("qk_norm_rope_append", 1, q, k, v, gamma_q, gamma_k, context_lens, block_table,
                         k_cache, v_cache, q_out, B, Hq, Hkv, D, page_size, max_pages, num_pages, rope_theta,
                         eps, stream);
}

int qk_norm_rope_append_multi(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                              const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                              const int32_t *context_lens, const int32_t *block_table,
                              pgqa_bf16 *k_cache, pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int M,
                              int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                              float rope_theta, float eps, cudaStream_t stream)
{
    return prologue_impl("qk_norm_rope_append_multi", M, q, k, v, gamma_q, gamma_k, context_lens, block_table,
                         k_cache, v_cache, q_out, B, Hq, Hkv, D, page_size, max_pages, num_pages, rope_theta,
                         eps, stream);
}

int decode_attn_partition_count(int B, int Hkv, int page_size, int max_pages, int num_partitions)
{
    if (B < 0 || Hkv <= 0 || page_size <= 0 || max_pages < 0 || num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "decode_attn_partition_count: invalid arguments");
    return pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                   sm_count_current_device());
}

size_t decode_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                  int num_partitions)
{
    (void)D;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || max_pages < 0 || num_partitions < 0)
        return 0;
    const int np = pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                           sm_count_current_device());
    return pgqa::decode_workspace_bytes(B, Hkv, Hq, np);
}

static int attn_impl(const char *fn, int M, const pgqa_bf16 *q, const pgqa_bf16 *k_cache, const pgqa_bf16 *v_cache,
                      const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages, int num_pages, float scale,
                      int num_partitions, float *out_f32, pgqa_bf16 *out_bf16, void *workspace,
                      size_t ws_bytes, cudaStream_t stream)
{
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (int st = check_pages(fn, page_size, max_pages, num_pages))
        return st;
    if (num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: num_partitions must be >= 0", fn);
    if (M < 1)
        return fail(PGQA_ERR_INVALID_ARG, "%s: M = %d new tokens per sequence, need >= 1", fn, M);
    if (M * (Hq / Hkv) > pgqa::kMaxGroupHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: M * (Hq / Hkv) = %d exceeds %d", fn, M * (Hq / Hkv),
                    pgqa::kMaxGroupHost);
    if (!std::isfinite(scale))
        return fail(PGQA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (static_cast<long long>(num_pages) * Hkv * page_size > 0x7FFFFFFFLL)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: num_pages * Hkv * page_size exceeds 2^31 - 1 rows", fn);
    if (B == 0)
        return ok();
    if (!q || !k_cache || !v_cache || !block_table || !context_lens)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!out_f32 && !out_bf16)
        return fail(PGQA_ERR_INVALID_ARG, "%s: out_f32 and out_bf16 are both NULL", fn);
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) ||
        !aligned4(block_table) || !aligned4(context_lens) || (workspace && !aligned16(workspace)))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte and index arrays 4-byte alignment", fn);
    const int np = pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                           sm_count_current_device());
    const size_t need = pgqa::decode_workspace_bytes(B, Hkv, M * Hq, np);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(PGQA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed for %d partitions, got %zu",
                    fn, need, np, workspace ? ws_bytes : static_cast<size_t>(0));
    pgqa::DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.scale = scale;
    a.num_partitions = np;
    a.pages_per_part = max_pages > 0 ? (max_pages + np - 1) / np : 1;
    a.out_f32 = out_f32;
    a.out_bf16 = out_bf16;
    a.ws = static_cast<float *>(workspace);
    a.M = M;
    a.sm_count = sm_count_current_device();
    cudaError_t err = pgqa::launch_decode(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int decode_attn_paged(const pgqa_bf16 *q, const pgqa_bf16 *k_cache, const pgqa_bf16 *v_cache,
                      const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages, int num_pages, float scale,
                      int num_partitions, float *out_f32, pgqa_bf16 *out_bf16, void *workspace,
                      size_t ws_bytes, cudaStream_t stream)
{
    return attn_impl("decode_attn_paged", 1, q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
                     page_size, max_pages, num_pages, scale, num_partitions, out_f32, out_bf16, workspace,
                     ws_bytes, stream);
}

int decode_attn_paged_multi(const pgqa_bf16 *q, const pgqa_bf16 *k_cache, const pgqa_bf16 *v_cache,
                            const int32_t *block_table, const int32_t *context_lens, int B, int M,
                            int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                            float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                            void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    return attn_impl("decode_attn_paged_multi", M, q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv,
                     D, page_size, max_pages, num_pages, scale, num_partitions, out_f32, out_bf16, workspace,
                     ws_bytes, stream);
}

size_t decode_attn_multi_workspace_size(int B, int M, int Hq, int Hkv, int D, int page_size, int max_pages,
                                        int num_partitions)
{
    if (M < 1)
        return 0;
    return decode_attn_workspace_size(B, M * Hq, Hkv, D, page_size, max_pages, num_partitions);
}

static int step_impl(const char *fn, int M, const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                      const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                      const int32_t *context_lens, const int32_t *block_table, pgqa_bf16 *k_cache,
                      pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D,
                      int page_size, int max_pages, int num_pages, float rope_theta, float eps,
                      float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                      void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (int st = check_pages(fn, page_size, max_pages, num_pages))
        return st;
    if (num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: num_partitions must be >= 0", fn);
    if (M < 1)
        return fail(PGQA_ERR_INVALID_ARG, "%s: M = %d new tokens per sequence, need >= 1", fn, M);
    if (M * (Hq / Hkv) > pgqa::kMaxGroupHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: M * (Hq / Hkv) = %d exceeds %d", fn, M * (Hq / Hkv),
                    pgqa::kMaxGroupHost);
    if (!std::isfinite(scale))
        return fail(PGQA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (!(rope_theta > 0.f) || !std::isfinite(rope_theta) || !(eps >= 0.f) || !std::isfinite(eps))
        return fail(PGQA_ERR_INVALID_ARG, "%s: rope_theta must be > 0 and eps >= 0", fn);
    if (static_cast<long long>(num_pages) * Hkv * page_size > 0x7FFFFFFFLL)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: num_pages * Hkv * page_size exceeds 2^31 - 1 rows", fn);
    if (B == 0)
        return ok();
    if (!q || !k || !v || !gamma_q || !gamma_k || !context_lens || !block_table || !k_cache ||
        !v_cache)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!out_f32 && !out_bf16)
        return fail(PGQA_ERR_INVALID_ARG, "%s: out_f32 and out_bf16 are both NULL", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gamma_q) ||
        !aligned16(gamma_k) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (q_out && !aligned16(q_out)) || (out_f32 && !aligned16(out_f32)) ||
        (out_bf16 && !aligned16(out_bf16)) || !aligned4(context_lens) || !aligned4(block_table) ||
        (workspace && !aligned16(workspace)))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte and index arrays 4-byte alignment", fn);
    const int np = pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                           sm_count_current_device());
    const size_t need = pgqa::decode_workspace_bytes(B, Hkv, M * Hq, np);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(PGQA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed for %d partitions, got %zu",
                    fn, need, np, workspace ? ws_bytes : static_cast<size_t>(0));
    pgqa::DecodeArgs a{};
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.scale = scale;
    a.num_partitions = np;
    a.pages_per_part = max_pages > 0 ? (max_pages + np - 1) / np : 1;
    a.out_f32 = out_f32;
    a.out_bf16 = out_bf16;
    a.ws = static_cast<float *>(workspace);
    a.fused = true;
    a.M = M;
    a.sm_count = sm_count_current_device();
    a.q_raw = q;
    a.k_new = k;
    a.v_new = v;
    a.gamma_q = gamma_q;
    a.gamma_k = gamma_k;
    a.q_out = q_out;
    a.rope_theta = static_cast<double>(rope_theta);
    a.eps = eps;
    cudaError_t err = pgqa::launch_decode(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int decode_step_paged(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                      const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                      const int32_t *context_lens, const int32_t *block_table, pgqa_bf16 *k_cache,
                      pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D,
                      int page_size, int max_pages, int num_pages, float rope_theta, float eps,
                      float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                      void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    return step_impl("decode_step_paged", 1, q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache,
                     v_cache, q_out, B, Hq, Hkv, D, page_size, max_pages, num_pages, rope_theta, eps, scale,
                     num_partitions, out_f32, out_bf16, workspace, ws_bytes, stream);
}

int decode_step_paged_multi(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                            const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                            const int32_t *context_lens, const int32_t *block_table, pgqa_bf16 *k_cache,
                            pgqa_bf16 *v_cache, pgqa_bf16 *q_out, int B, int M, int Hq, int Hkv, int D,
                            int page_size, int max_pages, int num_pages, float rope_theta, float eps,
                            float scale, int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                            void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    return step_impl("decode_step_paged_multi", M, q, k, v, gamma_q, gamma_k, context_lens, block_table,
                     k_cache, v_cache, q_out, B, Hq, Hkv, D, page_size, max_pages, num_pages, rope_theta, eps,
                     scale, num_partitions, out_f32, out_bf16, workspace, ws_bytes, stream);
}

int attn_partition_merge(const float *m, const float *l, const float *acc, int B, int Hq, int D,
                         int NP, float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream)
{
    const char *fn = "attn_partition_merge";
    if (B < 0 || Hq <= 0 || NP < 1)
        return fail(PGQA_ERR_INVALID_ARG, "%s: need B >= 0, Hq > 0, NP >= 1", fn);
    if (NP > pgqa::kMaxPartitions)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: NP = %d exceeds %d", fn, NP, pgqa::kMaxPartitions);
    if (D != pgqa::kHeadDimHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: head dim %d unsupported (only 128)", fn, D);
    if (static_cast<long long>(B) * Hq > 0x7FFFFFFFLL)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: B * Hq too large", fn);
    if (B == 0)
        return ok();
    if (!m || !l || !acc || (!out_f32 && !out_bf16))
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned4(m) || !aligned4(l) || !aligned16(acc) || (out_f32 && !aligned16(out_f32)) ||
        (out_bf16 && !aligned16(out_bf16)))
        return fail(PGQA_ERR_MISALIGNED, "%s: acc/out need 16-byte, m/l 4-byte alignment", fn);
    pgqa::MergeArgs a{};
    a.m = m;
    a.l = l;
    a.acc = acc;
    a.B = B;
    a.Hq = Hq;
    a.NP = NP;
    a.out_f32 = out_f32;
    a.out_bf16 = out_bf16;
    cudaError_t err = pgqa::launch_merge(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int attn_tile_init(float *m, float *l, float *acc, int B, int Hq, int D, cudaStream_t stream)
{
    const char *fn = "attn_tile_init";
    if (B < 0 || Hq <= 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: need B >= 0, Hq > 0", fn);
    if (D != pgqa::kHeadDimHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: head dim %d unsupported (only 128)", fn, D);
    if (B == 0)
        return ok();
    if (!m || !l || !acc)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned4(m) || !aligned4(l) || !aligned16(acc))
        return fail(PGQA_ERR_MISALIGNED, "%s: acc needs 16-byte, m/l 4-byte alignment", fn);
    cudaError_t err = pgqa::launch_tile_init(m, l, acc, B, Hq, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int attn_tile_update(const pgqa_bf16 *q, const pgqa_bf16 *k_tile, const pgqa_bf16 *v_tile,
                     int n_pos, int B, int Hq, int Hkv, int D, float scale, float *m, float *l,
                     float *acc, cudaStream_t stream)
{
    const char *fn = "attn_tile_update";
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (n_pos < 0 || n_pos > 512)
        return fail(PGQA_ERR_INVALID_ARG, "%s: n_pos = %d outside [0, 512]", fn, n_pos);
    if (!std::isfinite(scale))
        return fail(PGQA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (B == 0 || n_pos == 0)
        return ok();
    if (!q || !k_tile || !v_tile || !m || !l || !acc)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned16(q) || !aligned16(k_tile) || !aligned16(v_tile) || !aligned4(m) || !aligned4(l) ||
        !aligned16(acc))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte, m/l 4-byte alignment", fn);
    pgqa::TileArgs a{q, k_tile, v_tile, n_pos, B, Hq, Hkv, scale, m, l, acc, n_pos};
    cudaError_t err = pgqa::launch_tile_update(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int attn_tile_finalize(const float *m, const float *l, const float *acc, int B, int Hq, int D,
                       float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream)
{
    const char *fn = "attn_tile_finalize";
    if (B < 0 || Hq <= 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: need B >= 0, Hq > 0", fn);
    if (D != pgqa::kHeadDimHost)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: head dim %d unsupported (only 128)", fn, D);
    if (B == 0)
        return ok();
    if (!l || !acc || (!out_f32 && !out_bf16))
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned4(l) || !aligned16(acc) || (out_f32 && !aligned16(out_f32)) ||
        (out_bf16 && !aligned16(out_bf16)))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte, l 4-byte alignment", fn);
    cudaError_t err = pgqa::launch_tile_finalize(m, l, acc, B, Hq, out_f32, out_bf16, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

// The host-tiled pipeline; trace (n_trace copy groups, 4 events each) may
// be NULL.
static int host_tiled_impl(const char *fn, const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v,
                           int T, int B, int Hq, int Hkv, int D, float scale, int tile_len, int tiles_per_copy,
                           int n_slots, pgqa_bf16 *const *k_slots, pgqa_bf16 *const *v_slots,
                           cudaEvent_t const *events, float *m, float *l, float *acc, float *out_f32,
                           pgqa_bf16 *out_bf16, cudaStream_t compute_stream, cudaStream_t copy_stream,
                           cudaEvent_t const *trace, long n_trace)
{
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (T < 0 || tile_len < 1 || tile_len > 512 || n_slots < 2 || n_slots > 8 || tiles_per_copy < 1 ||
        tiles_per_copy > 64)
        return fail(PGQA_ERR_INVALID_ARG,
                    "%s: need T >= 0, tile_len in [1, 512], tiles_per_copy in [1, 64], n_slots in [2, 8]", fn);
    if (compute_stream == copy_stream)
        return fail(PGQA_ERR_INVALID_ARG, "%s: compute and copy streams must differ", fn);
    if (B == 0)
        return ok();
    if (!q || (T > 0 && (!host_k || !host_v)) || !k_slots || !v_slots || !events || !m || !l ||
        !acc || (!out_f32 && !out_bf16))
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    for (int s = 0; s < n_slots; ++s) {
        if (!k_slots[s] || !v_slots[s] || !events[s] || !events[n_slots + s])
            return fail(PGQA_ERR_INVALID_ARG, "%s: slot %d has a NULL buffer or event", fn, s);
        if (!aligned16(k_slots[s]) || !aligned16(v_slots[s]))
            return fail(PGQA_ERR_MISALIGNED, "%s: slot %d is not 16-byte aligned", fn, s);
    }
    if (!aligned16(q) || !aligned16(host_k) || !aligned16(host_v))
        return fail(PGQA_ERR_MISALIGNED, "%s: q and the host K/V need 16-byte alignment", fn);

    int st = attn_tile_init(m, l, acc, B, Hq, D, compute_stream);
    if (st != PGQA_OK)
        return st;
    const cudaEvent_t *copy_done = events;
    const cudaEvent_t *compute_done = events + n_slots;
    cudaError_t err;
    // No copy may land in a slot before the compute stream's earlier work
    // (which may still read the slots) is done.
    if ((err = cudaEventRecord(compute_done[0], compute_stream)) != cudaSuccess ||
        (err = cudaStreamWaitEvent(copy_stream, compute_done[0], 0)) != cudaSuccess)
        return cuda_fail(err, "attn_host_tiled_run: initial stream ordering");
    const size_t pos_bytes = static_cast<size_t>(Hkv) * D * sizeof(pgqa_bf16);
    // A copy fills a slot with up to tiles_per_copy consecutive tiles (one
    // transfer per slot and tensor: large copies reach the link's rate, 1 MiB
    // ones about half of it); the tiles are then updated one at a time.
    const long span_len = static_cast<long>(tiles_per_copy) * tile_len;
    const long n_copies = (static_cast<long>(T) + span_len - 1) / span_len;
    for (long g = 0; g < n_copies; ++g) {
        const int s = static_cast<int>(g % n_slots);
        const int t0 = static_cast<int>(g * span_len);
        const int n_span = T - t0 < span_len ? T - t0 : static_cast<int>(span_len);
        // The slot is free once the updates that last read it have finished.
        if (g >= n_slots && (err = cudaStreamWaitEvent(copy_stream, compute_done[s], 0)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: cudaStreamWaitEvent(copy)");
        const bool traced = trace && g < n_trace;
        if (traced && (err = cudaEventRecord(trace[4 * g], copy_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: trace event (copy start)");
        // Host rows of sequence b are [b][t0 .. t0+n_span); the slot holds
        // [b][0 .. n_span) packed: a 2-D copy with one row per sequence.
        const size_t row_bytes = static_cast<size_t>(n_span) * pos_bytes;
        const size_t src_pitch = static_cast<size_t>(T) * pos_bytes;
        const size_t dst_pitch = row_bytes;
        const char *hk = reinterpret_cast<const char *>(host_k) + static_cast<size_t>(t0) * pos_bytes;
        const char *hv = reinterpret_cast<const char *>(host_v) + static_cast<size_t>(t0) * pos_bytes;
        if (B == 1) {
            err = cudaMemcpyAsync(k_slots[s], hk, row_bytes, cudaMemcpyHostToDevice, copy_stream);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(v_slots[s], hv, row_bytes, cudaMemcpyHostToDevice, copy_stream);
        } else {
            err = cudaMemcpy2DAsync(k_slots[s], dst_pitch, hk, src_pitch, row_bytes, B,
                                    cudaMemcpyHostToDevice, copy_stream);
            if (err == cudaSuccess)
                err = cudaMemcpy2DAsync(v_slots[s], dst_pitch, hv, src_pitch, row_bytes, B,
                                        cudaMemcpyHostToDevice, copy_stream);
        }
        if (err != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: tile copy");
        if (traced && (err = cudaEventRecord(trace[4 * g + 1], copy_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: trace event (copy end)");
        if ((err = cudaEventRecord(copy_done[s], copy_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: cudaEventRecord(copy)");
        if ((err = cudaStreamWaitEvent(compute_stream, copy_done[s], 0)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: cudaStreamWaitEvent(compute)");
        if (traced && (err = cudaEventRecord(trace[4 * g + 2], compute_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: trace event (update start)");
        for (int p0 = 0; p0 < n_span; p0 += tile_len) {
            const size_t off = static_cast<size_t>(p0) * Hkv * D;
            pgqa::TileArgs a{q, k_slots[s] + off, v_slots[s] + off, n_span - p0 < tile_len ? n_span - p0 : tile_len,
                             B, Hq, Hkv, scale, m, l, acc, n_span};
            if ((err = pgqa::launch_tile_update(a, compute_stream)) != cudaSuccess)
                return cuda_fail(err, "attn_host_tiled_run: tile update");
        }
        if (traced && (err = cudaEventRecord(trace[4 * g + 3], compute_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: trace event (update end)");
        if ((err = cudaEventRecord(compute_done[s], compute_stream)) != cudaSuccess)
            return cuda_fail(err, "attn_host_tiled_run: cudaEventRecord(compute)");
    }
    return attn_tile_finalize(m, l, acc, B, Hq, D, out_f32, out_bf16, compute_stream);
}

int attn_host_tiled_run(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v,
                        int T, int B, int Hq, int Hkv, int D, float scale, int tile_len,
                        int tiles_per_copy, int n_slots, pgqa_bf16 *const *k_slots,
                        pgqa_bf16 *const *v_slots, cudaEvent_t const *events, float *m, float *l,
                        float *acc, float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t compute_stream,
                        cudaStream_t copy_stream)
{
    return host_tiled_impl("attn_host_tiled_run", q, host_k, host_v, T, B, Hq, Hkv, D, scale, tile_len,
                           tiles_per_copy, n_slots, k_slots, v_slots, events, m, l, acc, out_f32, out_bf16,
                           compute_stream, copy_stream, nullptr, 0);
}

int attn_host_tiled_run_traced(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v, int T,
                               int B, int Hq, int Hkv, int D, float scale, int tile_len, int tiles_per_copy,
                               int n_slots, pgqa_bf16 *const *k_slots, pgqa_bf16 *const *v_slots,
                               cudaEvent_t const *events, float *m, float *l, float *acc, float *out_f32,
                               pgqa_bf16 *out_bf16, cudaStream_t compute_stream, cudaStream_t copy_stream,
                               cudaEvent_t const *trace_events, int n_trace_groups)
{
    const char *fn = "attn_host_tiled_run_traced";
    if (n_trace_groups < 0 || (n_trace_groups > 0 && !trace_events))
        return fail(PGQA_ERR_INVALID_ARG, "%s: trace_events must hold 4 * n_trace_groups events", fn);
    for (int i = 0; i < 4 * n_trace_groups; ++i)
        if (!trace_events[i])
            return fail(PGQA_ERR_INVALID_ARG, "%s: trace event %d is NULL", fn, i);
    return host_tiled_impl(fn, q, host_k, host_v, T, B, Hq, Hkv, D, scale, tile_len, tiles_per_copy, n_slots,
                           k_slots, v_slots, events, m, l, acc, out_f32, out_bf16, compute_stream, copy_stream,
                           trace_events, n_trace_groups);
}

int attn_host_direct_partition_count(int B, int Hkv, int T, int num_partitions)
{
    if (B < 0 || Hkv <= 0 || T < 0 || num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "attn_host_direct_partition_count: bad sizes");
    return pgqa::host_direct_partitions(B, Hkv, T, num_partitions, sm_count_current_device());
}

size_t attn_host_direct_workspace_size(int B, int Hq, int Hkv, int T, int num_partitions)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || num_partitions < 0)
        return 0;
    const int np = pgqa::host_direct_partitions(B, Hkv, T, num_partitions, sm_count_current_device());
    return pgqa::host_direct_workspace_bytes(B, Hq, np);
}

int attn_host_direct(const pgqa_bf16 *q, const pgqa_bf16 *host_k, const pgqa_bf16 *host_v, int T,
                     int B, int Hq, int Hkv, int D, float scale, int num_partitions, float *out_f32,
                     pgqa_bf16 *out_bf16, void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    const char *fn = "attn_host_direct";
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (T < 0 || num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: need T >= 0 and num_partitions >= 0", fn);
    if (!std::isfinite(scale))
        return fail(PGQA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (static_cast<long long>(B) * T * Hkv > (1LL << 40))
        return fail(PGQA_ERR_UNSUPPORTED, "%s: B * T * Hkv too large", fn);
    if (B == 0)
        return ok();
    if (!q || (T > 0 && (!host_k || !host_v)) || (!out_f32 && !out_bf16))
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned16(q) || (out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) ||
        !aligned16(host_k) || !aligned16(host_v) || (workspace && !aligned16(workspace)))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte alignment", fn);
    // The history must be pinned host memory mapped into the device address
    // space; its device-side address is what the kernel reads through.
    void *dk = nullptr, *dv = nullptr;
    if (T > 0) {
        if (cudaHostGetDevicePointer(&dk, const_cast<pgqa_bf16 *>(host_k), 0) != cudaSuccess ||
            cudaHostGetDevicePointer(&dv, const_cast<pgqa_bf16 *>(host_v), 0) != cudaSuccess || !dk || !dv) {
            cudaGetLastError();
            return fail(PGQA_ERR_INVALID_ARG, "%s: host_k / host_v are not mapped pinned host memory", fn);
        }
    }
    const int np = pgqa::host_direct_partitions(B, Hkv, T, num_partitions, sm_count_current_device());
    const size_t need = pgqa::host_direct_workspace_bytes(B, Hq, np);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(PGQA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed for %d partitions, got %zu", fn,
                    need, np, workspace ? ws_bytes : static_cast<size_t>(0));
    pgqa::HostDirectArgs a{};
    a.q = q;
    a.k = static_cast<const pgqa_bf16 *>(dk);
    a.v = static_cast<const pgqa_bf16 *>(dv);
    a.T = T;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.scale = scale;
    a.num_partitions = np;
    a.out_f32 = out_f32;
    a.out_bf16 = out_bf16;
    a.ws = static_cast<float *>(workspace);
    cudaError_t err = pgqa::launch_host_direct(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}


int qk_norm_rope_append_int8(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                             const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                             const int32_t *context_lens, const int32_t *block_table, int8_t *k_cache8,
                             int8_t *v_cache8, float *k_scale, float *v_scale, pgqa_bf16 *q_out, int B,
                             int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                             float rope_theta, float eps, cudaStream_t stream)
{
    const char *fn = "qk_norm_rope_append_int8";
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (int st = check_pages(fn, page_size, max_pages, num_pages))
        return st;
    if (!(rope_theta > 0.f) || !std::isfinite(rope_theta) || !(eps >= 0.f) || !std::isfinite(eps))
        return fail(PGQA_ERR_INVALID_ARG, "%s: rope_theta must be > 0 and eps >= 0", fn);
    if (B == 0)
        return ok();
    if (!q || !k || !v || !gamma_q || !gamma_k || !context_lens || !block_table || !k_cache8 || !v_cache8 ||
        !k_scale || !v_scale || !q_out)
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(gamma_q) || !aligned16(gamma_k) ||
        !aligned16(k_cache8) || !aligned16(v_cache8) || !aligned16(k_scale) || !aligned16(v_scale) ||
        !aligned16(q_out) || !aligned4(context_lens) || !aligned4(block_table))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte and index arrays 4-byte alignment", fn);
    pgqa::PrologueArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.gamma_q = gamma_q;
    a.gamma_k = gamma_k;
    a.context_lens = context_lens;
    a.block_table = block_table;
    a.q_out = q_out;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.rope_theta = static_cast<double>(rope_theta);
    a.eps = eps;
    a.M = 1;
    a.k_cache8 = k_cache8;
    a.v_cache8 = v_cache8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t err = pgqa::launch_prologue(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

size_t decode_attn_int8_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                       int num_partitions)
{
    (void)D;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || max_pages < 0 || num_partitions < 0)
        return 0;
    const int np = pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                           sm_count_current_device());
    return pgqa::decode_int8_workspace_bytes(B, Hkv, Hq, np);
}

// Validation, partition choice and launch shared by decode_attn_paged_int8
// (fused = false: q is the rotated query) and decode_step_paged_int8 (fused:
// q, k, v are the new token's raw heads and the kernel appends to the cache).
static int int8_attn_impl(const char *fn, bool fused, const pgqa_bf16 *q, const pgqa_bf16 *k,
                          const pgqa_bf16 *v, const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k,
                          const int8_t *k_cache8, const int8_t *v_cache8, const float *k_scale,
                          const float *v_scale, const int32_t *block_table, const int32_t *context_lens,
                          pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                          int num_pages, float rope_theta, float eps, float scale, int num_partitions,
                          float *out_f32, pgqa_bf16 *out_bf16, void *workspace, size_t ws_bytes,
                          cudaStream_t stream)
{
    if (int st = check_heads(fn, B, Hq, Hkv, D))
        return st;
    if (int st = check_pages(fn, page_size, max_pages, num_pages))
        return st;
    if (num_partitions < 0)
        return fail(PGQA_ERR_INVALID_ARG, "%s: num_partitions must be >= 0", fn);
    if (!std::isfinite(scale))
        return fail(PGQA_ERR_INVALID_ARG, "%s: scale is not finite", fn);
    if (fused && (!(rope_theta > 0.f) || !std::isfinite(rope_theta) || !(eps >= 0.f) || !std::isfinite(eps)))
        return fail(PGQA_ERR_INVALID_ARG, "%s: rope_theta must be > 0 and eps >= 0", fn);
    if (static_cast<long long>(num_pages) * Hkv * page_size > 0x7FFFFFFFLL)
        return fail(PGQA_ERR_UNSUPPORTED, "%s: num_pages * Hkv * page_size exceeds 2^31 - 1 rows", fn);
    if (B == 0)
        return ok();
    if (!q || !k_cache8 || !v_cache8 || !k_scale || !v_scale || !block_table || !context_lens ||
        (fused && (!k || !v || !gamma_q || !gamma_k)))
        return fail(PGQA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    if (!out_f32 && !out_bf16)
        return fail(PGQA_ERR_INVALID_ARG, "%s: out_f32 and out_bf16 are both NULL", fn);
    if (!aligned16(q) || !aligned16(k_cache8) || !aligned16(v_cache8) || !aligned16(k_scale) ||
        !aligned16(v_scale) || (out_f32 && !aligned16(out_f32)) || (out_bf16 && !aligned16(out_bf16)) ||
        !aligned4(block_table) || !aligned4(context_lens) || (workspace && !aligned16(workspace)) ||
        (fused && (!aligned16(k) || !aligned16(v) || !aligned16(gamma_q) || !aligned16(gamma_k) ||
                   (q_out && !aligned16(q_out)))))
        return fail(PGQA_ERR_MISALIGNED, "%s: tensors need 16-byte and index arrays 4-byte alignment", fn);
    const int np = pgqa::choose_partitions(B, Hkv, page_size, max_pages, num_partitions,
                                           sm_count_current_device());
    const size_t need = pgqa::decode_int8_workspace_bytes(B, Hkv, Hq, np);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(PGQA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed for %d partitions, got %zu", fn, need,
                    np, workspace ? ws_bytes : static_cast<size_t>(0));
    pgqa::DecodeInt8Args a{};
    a.q = q;
    a.k_cache8 = k_cache8;
    a.v_cache8 = v_cache8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.scale = scale;
    a.num_partitions = np;
    a.pages_per_part = max_pages > 0 ? (max_pages + np - 1) / np : 1;
    a.out_f32 = out_f32;
    a.out_bf16 = out_bf16;
    a.ws = static_cast<float *>(workspace);
    if (fused) {
        a.fused = true;
        a.q_raw = q;
        a.k_new = k;
        a.v_new = v;
        a.gamma_q = gamma_q;
        a.gamma_k = gamma_k;
        a.q_out = q_out;
        a.rope_theta = static_cast<double>(rope_theta);
        a.eps = eps;
    }
    a.sm_count = sm_count_current_device();
    cudaError_t err = pgqa::launch_decode_int8(a, stream);
    if (err != cudaSuccess)
        return cuda_fail(err, fn);
    return ok();
}

int decode_attn_paged_int8(const pgqa_bf16 *q, const int8_t *k_cache8, const int8_t *v_cache8,
                           const float *k_scale, const float *v_scale, const int32_t *block_table,
                           const int32_t *context_lens, int B, int Hq, int Hkv, int D, int page_size,
                           int max_pages, int num_pages, float scale, int num_partitions, float *out_f32,
                           pgqa_bf16 *out_bf16, void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    return int8_attn_impl("decode_attn_paged_int8", false, q, nullptr, nullptr, nullptr, nullptr, k_cache8,
                          v_cache8, k_scale, v_scale, block_table, context_lens, nullptr, B, Hq, Hkv, D,
                          page_size, max_pages, num_pages, 1.0f, 0.0f, scale, num_partitions, out_f32, out_bf16,
                          workspace, ws_bytes, stream);
}

int decode_step_paged_int8(const pgqa_bf16 *q, const pgqa_bf16 *k, const pgqa_bf16 *v,
                           const pgqa_bf16 *gamma_q, const pgqa_bf16 *gamma_k, const int32_t *context_lens,
                           const int32_t *block_table, int8_t *k_cache8, int8_t *v_cache8, float *k_scale,
                           float *v_scale, pgqa_bf16 *q_out, int B, int Hq, int Hkv, int D, int page_size,
                           int max_pages, int num_pages, float rope_theta, float eps, float scale,
                           int num_partitions, float *out_f32, pgqa_bf16 *out_bf16, void *workspace,
                           size_t ws_bytes, cudaStream_t stream)
{
    return int8_attn_impl("decode_step_paged_int8", true, q, k, v, gamma_q, gamma_k, k_cache8, v_cache8, k_scale,
                          v_scale, block_table, context_lens, q_out, B, Hq, Hkv, D, page_size, max_pages,
                          num_pages, rope_theta, eps, scale, num_partitions, out_f32, out_bf16, workspace,
                          ws_bytes, stream);
}

} // extern "C"
