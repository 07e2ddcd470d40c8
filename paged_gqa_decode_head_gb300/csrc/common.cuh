// common.cuh -- device helpers shared by the libpgqa kernels (sm_103a).
//
// bf16 unpacking, 16-byte shared/global loads, mbarrier and bulk-copy (TMA)
// wrappers written as inline PTX, and the bounded wait used by every
// asynchronous copy.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pgqa.h"

namespace pgqa {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 8;
constexpr int kChunkTokens = 16;                      // keys per staged chunk
constexpr int kRowBytes = kHeadDim * 2;               // one bf16 D-vector
constexpr int kChunkBytes = kChunkTokens * kRowBytes; // 4 KiB of K (or V)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kEmptyMax = -1e30f; // start value of the running max

// A wait on an asynchronous copy gives up after this long and raises
// PGQA_DEVERR_WAIT_TIMEOUT instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;

// ---------------------------------------------------------------- bf16
// bf16 is the top half of a binary32, so widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &u, float *f)
{
    f[0] = bf16_lo(u.x), f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y), f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z), f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w), f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x)
{
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
}

// ---------------------------------------------------------------- memory
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream128(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier / bulk copy
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy accesses of shared memory before later
// async-proxy writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy view of global memory before its
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return true;
}

// L2 policy for data that is read exactly once (streamed KV).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`. Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
                 : "memory");
}


// As bulk_copy_g2s, with the default L2 policy.
__device__ __forceinline__ void bulk_copy_g2s_nohint(void *dst, const void *src, uint32_t bytes,
                                                     uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// ---------------------------------------------------------------- 2-D TMA
// Tiled TMA load of box {x, y} of a 2-D tensor map into this CTA's shared
// memory, completing its bytes on `bar`. x * element size must be a multiple
// of 16 bytes; dst must be aligned to the map's swizzle atom (1024 B for
// 128-byte swizzle).
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
                 : "memory");
}

// Tiled TMA load of box {x, y, z} of a 3-D tensor map (same rules as 2-D).
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
                 "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- warp MMA
// Four 8x8 b16 matrices from shared memory; lane L gives the address of row
// L % 8 of matrix L / 8; register q receives matrix q in mma fragment order.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// Same, each matrix transposed on the way.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// d += A (16x16, row) * B (16x8, col), bf16 inputs, fp32 accumulate. Only
// the fragments of A rows 0..7 are passed (rows 8..15 are zero).
__device__ __forceinline__ void mma_bf16_rows8(float (&d)[4], uint32_t a_lo_k, uint32_t a_hi_k,
                                               uint32_t b0, uint32_t b1)
{
    const uint32_t zero = 0;
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a_lo_k), "r"(zero), "r"(a_hi_k), "r"(zero), "r"(b0), "r"(b1));
}

// d += A (16x16, row) * B (16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// As mma_bf16_16816 with fp16 A and B operands.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two int8 bytes of `bytes` (selected by `sel`: byte index of the low half
// in bits 0-3, of the high half in bits 8-11) -> fp16x2, exactly: the biased
// byte b + 128 becomes the mantissa of 1024 (fp16 0x6400 | byte), and 1152 is
// subtracted.
__device__ __forceinline__ uint32_t int8x2_to_f16x2(uint32_t bytes, uint32_t sel)
{
    const uint32_t biased = bytes ^ 0x80808080u;
    const uint32_t h = __byte_perm(biased, 0x64646464u, sel | 0x4040u);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

// As int8x2_to_f16x2 on bytes already biased (xor 0x80808080), so that one
// bias serves the two halves taken from a register.
__device__ __forceinline__ uint32_t biased8x2_to_f16x2(uint32_t biased, uint32_t sel)
{
    const uint32_t h = __byte_perm(biased, 0x64646464u, sel | 0x4040u);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

// Two floats -> packed fp16x2 (nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t pair)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(pair & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t pair)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(pair >> 16)));
}

// Transpose an 8x8 b16 matrix held as an mma fragment (thread (g, t) holds
// row g, columns 2t and 2t+1) into the same fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// Two floats -> packed bf16x2 (nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Device-scope atomic add with release and acquire semantics.
__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned *addr, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(addr), "r"(v)
                 : "memory");
    return old;
}

// 32-bit global load kept where it is written, so that several independent
// loads issued one after another are in flight together.
__device__ __forceinline__ int ldg_i32_now(const int32_t *p)
{
    int v;
    asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Block until the grids this one depends on have completed and their memory
// is visible (no-op when launched without a programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void allow_dependent_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Timeline builds (-DPGQA_TIMELINE, a separate library made by the package's
// timeline module) stamp %globaltimer at each phase of the split kernels
// (bf16 and INT8; their parameter structs carry `tl` and `tl_launch`) into a
// caller buffer [launch][CTA][kTimelineSlots]; other builds compile the
// stamps out. Slots: 0 CTA start, 1 block-table entries in hand, 2 first
// requests issued, 3 grid dependency released, 4 query rotated (fused step),
// 5 a warp's second chunk landed, 6 last chunk landed (latest warp), 7 warp
// records merged, 8 partition state written, 9 ticket back, 10 merge done.
constexpr int kTimelineSlots = 12;
#ifdef PGQA_TIMELINE
// host side (decode.cu): the attached buffer and the next launch's slot
unsigned long long *timeline_buffer();
int timeline_next_launch();
#define TL_INDEX(slot)                                                                                       \
    ((static_cast<size_t>(p.tl_launch) * gridDim.x * gridDim.y * gridDim.z + blockIdx.x +                     \
      gridDim.x * (blockIdx.y + static_cast<size_t>(gridDim.y) * blockIdx.z)) *                                \
         kTimelineSlots +                                                                                     \
     (slot))
#define TL_STAMP(slot)                                                                                       \
    do {                                                                                                     \
        if (p.tl && threadIdx.x == 0)                                                                        \
            p.tl[TL_INDEX(slot)] = globaltimer_ns();                                                         \
    } while (0)
#define TL_STAMP_LATEST(slot)                                                                                \
    do {                                                                                                     \
        if (p.tl && (threadIdx.x & 31) == 0)                                                                 \
            atomicMax(&p.tl[TL_INDEX(slot)], globaltimer_ns());                                              \
    } while (0)
#else
#define TL_STAMP(slot) \
    do {               \
    } while (0)
#define TL_STAMP_LATEST(slot) \
    do {                      \
    } while (0)
#endif

} // namespace pgqa
