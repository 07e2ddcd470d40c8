// decode_static.cu -- decode_attn_paged_static: paged decode attention whose
// partition scratch lives in a fixed array inside this library, for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run attention: code inside a custom allocator or memory-pool
// callback, plugins of hosts that own every device allocation and hand out no
// scratch, hard real-time loops that forbid allocation after start-up. This
// entry point lets them run the split-KV path without passing a workspace.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes. Every
// GPU that loads this library holds it until the process exits. Host code
// cannot use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels as an ordinary pointer.
#include <mutex>

#include "launch.h"
#include "pgqa.h"

namespace {

constexpr size_t kStaticScratchBytes = PGQA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first call for that device.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (err != cudaSuccess)
            return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" int decode_attn_paged_static(const pgqa_bf16 *q, const pgqa_bf16 *k_cache,
                                        const pgqa_bf16 *v_cache, const int32_t *block_table,
                                        const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                        int page_size, int max_pages, int num_pages, float scale,
                                        int num_partitions, float *out_f32, pgqa_bf16 *out_bf16,
                                        cudaStream_t stream)
{
    const size_t need =
        decode_attn_workspace_size(B, Hq, Hkv, D, page_size, max_pages, num_partitions);
    if (need > kStaticScratchBytes)
        return pgqa::report_error(
            PGQA_ERR_WORKSPACE,
            "decode_attn_paged_static: these sizes need %zu bytes of scratch but the built-in "
            "array holds %zu; call decode_attn_paged with a workspace or ask for fewer partitions",
            need, kStaticScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        cudaError_t err = scratch_address(&scratch);
        if (err != cudaSuccess)
            return pgqa::report_error(PGQA_ERR_CUDA,
                                      "decode_attn_paged_static: cudaGetSymbolAddress failed: %s",
                                      cudaGetErrorString(err));
        // The array keeps whatever the last call left, and a call with other
        // sizes may have left partition data where this call's partition
        // tickets go; they must start at zero.
        if (B > 0 && Hkv > 0) {
            err = cudaMemsetAsync(scratch, 0, pgqa::decode_ticket_bytes(B, Hkv), stream);
            if (err != cudaSuccess)
                return pgqa::report_error(PGQA_ERR_CUDA, "decode_attn_paged_static: clearing tickets: %s",
                                          cudaGetErrorString(err));
        }
    }
    return decode_attn_paged(q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
                             page_size, max_pages, num_pages, scale, num_partitions, out_f32,
                             out_bf16, scratch, kStaticScratchBytes, stream);
}
