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
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress and passed to the kernels as an ordinary pointer. The
// lookup is set-up work done once per device and context: the address is
// kept together with the unique id of the context it was found in
// (cuCtxGetId), so a context torn down and made again (cudaDeviceReset),
// which may load the array elsewhere, gets a fresh lookup instead of a stale
// address.
#include <mutex>

#include <cuda.h>

#include "launch.h"
#include "pgqa.h"

namespace {

constexpr size_t kStaticScratchBytes = PGQA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct ScratchSlot {
    unsigned long long ctx_id; // unique id of the context the address belongs to
    void *ptr;                 // device address of g_static_scratch there, or NULL
};

std::mutex g_setup_mutex;
ScratchSlot g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current context (false if there is none
// or the driver cannot say).
bool current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device. The first call
// on a device, and the first after its context was made again, looks it up.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    if (!known || !g_scratch[dev].ptr || g_scratch[dev].ctx_id != id) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_static_scratch); // also makes the context current if needed
        if (err != cudaSuccess)
            return err;
        if (!known && !current_context_id(&id))
            return cudaErrorNotSupported;
        g_scratch[dev] = ScratchSlot{id, p};
    }
    *out = g_scratch[dev].ptr;
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
                                      "decode_attn_paged_static: no device address for the scratch array: %s",
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
