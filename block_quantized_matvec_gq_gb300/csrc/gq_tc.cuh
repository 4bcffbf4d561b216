// gq_tc.cuh -- building blocks shared by the tensor-core (tcgen05) kernels:
// mbarriers with bounded waits, TMA and bulk copies, shared-memory matrix
// and instruction descriptors, MMA issue/commit, tensor-memory loads, the
// UMMA K-major no-swizzle operand layout, and host-side tensor maps.
#pragma once

#include <cuda.h>

#include <cstring>

#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {
namespace tcu {

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// A waiting thread may be suspended up to this long inside one try_wait
// (it resumes as soon as the phase completes), so waiting warps do not
// compete with working warps for issue slots.
constexpr uint32_t kSuspendNs = 20000;
// kCluster: acquire at cluster scope (arrivals from the peer CTA of a pair,
// or from a pair MMA's multicast commit).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if (kCluster)
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
    else
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
    return ok != 0;
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// Bounded wait for the phase of `bar` with the given parity.  Returns false
// (raising the CTA abort flag and the device status) on timeout, or when
// another role has already aborted.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort, int *status)
{
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait<kCluster>(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicExch(status, GQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// Warp-uniform form (all lanes agree).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort, int *status)
{
    return __all_sync(0xffffffffu, wait_bounded<kCluster>(bar, parity, abort, status));
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// tcgen05 shared-memory matrix descriptor, K-major, no swizzle: start
// address, LBO = byte stride between core matrices along K, SBO = byte
// stride between 8-row groups along M/N, descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B types at
// bits 7-9 and 10-12 (0 = f16, 1 = bf16; always the same for A and B),
// both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_f16(int m, int n, bool bf16)
{
    return (1u << 4) | (bf16 ? ((1u << 7) | (1u << 10)) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// Two CTAs of a cluster share one MMA: M = 256 (128 rows of A and of D per
// CTA, in each CTA's own shared and tensor memory at the same addresses),
// B split by N between the two CTAs' shared memory.  Rank 0 issues the MMAs.
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier given by its shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at offset `bar` of both CTAs of the pair when
// every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar)
{
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------- operand conversion
// Both operands of a 32-block are written as four 8-element K groups; inside
// a group the elements are stored in the order 0,4,1,5,2,6,3,7 (the order in
// which the nibble unpacking below produces them).  A and B use the same
// order, so the dot products are unchanged.
__device__ __forceinline__ uint4 nib8_to_f16(uint32_t w)
{
    const uint32_t w2 = w >> 8;
    uint32_t a0 = (w & 0x000F000Fu) | 0x64006400u;   // 1024 + (e0, e4)
    uint32_t a1 = (w & 0x00F000F0u) | 0x64006400u;   // 1024 + 16 (e1, e5)
    uint32_t a2 = (w2 & 0x000F000Fu) | 0x64006400u;  // 1024 + (e2, e6)
    uint32_t a3 = (w2 & 0x00F000F0u) | 0x64006400u;  // 1024 + 16 (e3, e7)
    const __half2 c1032 = __float2half2_rn(1032.0f);
    const __half2 c16 = __float2half2_rn(0.0625f);
    const __half2 c72 = __float2half2_rn(-72.0f);
    __half2 r0 = __hsub2(*reinterpret_cast<__half2 *>(&a0), c1032);
    __half2 r1 = __hfma2(*reinterpret_cast<__half2 *>(&a1), c16, c72);
    __half2 r2 = __hsub2(*reinterpret_cast<__half2 *>(&a2), c1032);
    __half2 r3 = __hfma2(*reinterpret_cast<__half2 *>(&a3), c16, c72);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t *>(&r0);
    o.y = *reinterpret_cast<uint32_t *>(&r1);
    o.z = *reinterpret_cast<uint32_t *>(&r2);
    o.w = *reinterpret_cast<uint32_t *>(&r3);
    return o;
}
// Eight int8 codes (two words, elements 0..3 and 4..7) -> f16 in group order.
__device__ __forceinline__ uint4 s8x8_to_f16(uint32_t lo, uint32_t hi)
{
    lo ^= 0x80808080u;  // offset binary: u = q + 128
    hi ^= 0x80808080u;
    const uint32_t t01 = __byte_perm(lo, hi, 0x5140);  // u0 u4 u1 u5
    const uint32_t t23 = __byte_perm(lo, hi, 0x7362);  // u2 u6 u3 u7
    uint32_t a0 = __byte_perm(t01, 0x64646464u, 0x4140);  // 1024 + (u0, u4)
    uint32_t a1 = __byte_perm(t01, 0x64646464u, 0x4342);  // 1024 + (u1, u5)
    uint32_t a2 = __byte_perm(t23, 0x64646464u, 0x4140);
    uint32_t a3 = __byte_perm(t23, 0x64646464u, 0x4342);
    const __half2 c = __float2half2_rn(1152.0f);
    __half2 r0 = __hsub2(*reinterpret_cast<__half2 *>(&a0), c);
    __half2 r1 = __hsub2(*reinterpret_cast<__half2 *>(&a1), c);
    __half2 r2 = __hsub2(*reinterpret_cast<__half2 *>(&a2), c);
    __half2 r3 = __hsub2(*reinterpret_cast<__half2 *>(&a3), c);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t *>(&r0);
    o.y = *reinterpret_cast<uint32_t *>(&r1);
    o.z = *reinterpret_cast<uint32_t *>(&r2);
    o.w = *reinterpret_cast<uint32_t *>(&r3);
    return o;
}
// Byte offset of (row, K group kg) in an operand stage: core matrix
// (row/8, kg) at ((row/8)*4 + kg)*128, row%8 at 16-byte steps inside it.
__device__ __forceinline__ uint32_t op_off(int row, int kg) { return (((row >> 3) * 4 + kg) << 7) + ((row & 7) << 4); }

}  // namespace tcu

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static inline EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D tensor [outer][inner] of `dt` elements with row stride `stride` bytes;
// box inner x outer elements; `sw` the shared-memory swizzle of the box.
static inline bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                     uint64_t stride, uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gq
