// launch.h -- host-side launchers of the libpgqa kernels (internal).
// The C ABI in api.cu validates arguments and then calls these.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "pgqa.h"

namespace pgqa {

struct PrologueArgs {
    const pgqa_bf16 *q, *k, *v, *gamma_q, *gamma_k;
    const int32_t *context_lens, *block_table;
    pgqa_bf16 *k_cache, *v_cache, *q_out;
    int B, Hq, Hkv, page_size, max_pages, num_pages;
    double rope_theta;
    float eps;
    int M; // new tokens per sequence, at positions T - M .. T - 1 (0 or 1: one)
    // INT8 cache instead of k_cache / v_cache when k_cache8 is set
    int8_t *k_cache8, *v_cache8;
    float *k_scale, *v_scale;
};

struct DecodeArgs {
    const pgqa_bf16 *q, *k_cache, *v_cache;
    const int32_t *block_table, *context_lens;
    int B, Hq, Hkv, page_size, max_pages, num_pages;
    float scale;
    int num_partitions;  // NP >= 1 (already resolved)
    int pages_per_part;  // ceil(max_pages / NP)
    float *out_f32;      // nullable
    pgqa_bf16 *out_bf16; // nullable
    float *ws;           // partial states when NP > 1
    int M; // new tokens (queries) per sequence; 0 or 1 = the single-token step
    int sm_count; // SMs of the device (selects the CTA shape)
    // fused decode step (qk_norm_rope_append + attention in one launch)
    bool fused;
    const pgqa_bf16 *q_raw, *k_new, *v_new, *gamma_q, *gamma_k;
    pgqa_bf16 *q_out; // nullable
    double rope_theta;
    float eps;
};

struct MergeArgs {
    const float *m, *l, *acc;
    int B, Hq, NP;
    int M; // query rows per sequence are M * Hq (0 or 1: one)
    float *out_f32;
    pgqa_bf16 *out_bf16;
    // When context_lens is non-null, sequence b uses only its first
    // ceil(ceil(T_b / page_size) / pages_per_part) partitions and m is in
    // base-2 units (the decode kernel's private workspace format).
    const int32_t *context_lens;
    int page_size, pages_per_part, max_pages;
};

struct TileArgs {
    const pgqa_bf16 *q, *k_tile, *v_tile;
    int n_pos, B, Hq, Hkv;
    float scale;
    float *m, *l, *acc;
    int seq_stride; // positions from one sequence's rows to the next's in the tile buffers (0: n_pos)
};

struct HostDirectArgs {
    const pgqa_bf16 *q, *k, *v; // k, v: device-side addresses of mapped host memory
    int T, B, Hq, Hkv;
    float scale;
    int num_partitions; // resolved, >= 1
    float *out_f32;
    pgqa_bf16 *out_bf16;
    float *ws; // partition states when num_partitions > 1
};

// Shortest partition of the zero-copy variant (positions).
constexpr int kHostDirectMinPositions = 512;

// Largest partition count the merge supports.
constexpr int kMaxPartitions = 65536;

cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t stream);
int host_direct_partitions(int B, int Hkv, int T, int requested, int sm_count);
size_t host_direct_workspace_bytes(int B, int Hq, int num_partitions);
cudaError_t launch_host_direct(const HostDirectArgs &a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t stream);
cudaError_t launch_tile_init(float *m, float *l, float *acc, int B, int Hq, cudaStream_t stream);
cudaError_t launch_tile_update(const TileArgs &a, cudaStream_t stream);
cudaError_t launch_tile_finalize(const float *m, const float *l, const float *acc, int B, int Hq,
                                 float *out_f32, pgqa_bf16 *out_bf16, cudaStream_t stream);

// Partition choice shared by decode_attn_paged and its workspace query.
int choose_partitions(int B, int Hkv, int page_size, int max_pages, int requested, int sm_count);
size_t decode_workspace_bytes(int B, int Hkv, int Hq, int num_partitions);
// Bytes at the start of that workspace holding the partition tickets.
size_t decode_ticket_bytes(int B, int Hkv);

// Each translation unit keeps its own sticky device flag word; these read
// (and optionally clear) it synchronously on the current device.
cudaError_t read_flags_prologue(unsigned *flags, bool clear);
cudaError_t read_flags_decode(unsigned *flags, bool clear);
cudaError_t launch_wait_selftest(cudaStream_t stream);

// Decode attention over an INT8 cache (decode_int8.cu).
struct DecodeInt8Args {
    const pgqa_bf16 *q;
    const int8_t *k_cache8, *v_cache8;
    const float *k_scale, *v_scale;
    const int32_t *block_table, *context_lens;
    int B, Hq, Hkv, page_size, max_pages, num_pages;
    float scale;
    int num_partitions, pages_per_part;
    float *out_f32;
    pgqa_bf16 *out_bf16;
    float *ws;
    int sm_count; // SMs of the device (selects the CTA shape)
    // fused decode step (decode_step_paged_int8): the prologue runs in the
    // attention kernel; q is unused, the caches are written
    bool fused;
    const pgqa_bf16 *q_raw, *k_new, *v_new, *gamma_q, *gamma_k;
    pgqa_bf16 *q_out;
    double rope_theta;
    float eps;
};
cudaError_t launch_decode_int8(const DecodeInt8Args &a, cudaStream_t stream);
size_t decode_int8_workspace_bytes(int B, int Hkv, int Hq, int num_partitions);
cudaError_t read_flags_int8(unsigned *flags, bool clear);

// Launch `kernel` on `stream` with programmatic stream serialisation: it may
// start while the previous kernel in the stream is still running, and must
// call griddepcontrol.wait before touching anything that kernel produces.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Record a message for pgqa_last_error() and return `code` (printf format).
int report_error(int code, const char *fmt, ...);

} // namespace pgqa
