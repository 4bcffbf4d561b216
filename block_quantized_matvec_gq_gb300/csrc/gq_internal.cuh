// gq_internal.cuh -- device helpers shared by the libgq kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gq.h"

namespace gq {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- launch
// Programmatic dependent launch: a kernel may start while the previous
// kernel in the stream drains; it reads its activation input only after
// griddepcontrol.wait (which returns once the previous grid's memory is
// visible), and lets the next kernel start early with launch_dependents.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- memory
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Streaming weight loads: read once, no L1 allocation.  (An L2 eviction
// hint is accepted by sm_103a only on the 32-byte form.)
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 32-byte load (two 16-byte halves), evict-first in L2.
__device__ __forceinline__ void ld_stream32(const void *p, uint4 &a, uint4 &b)
{
    asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ uint16_t ld_stream_u16(const void *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Prefetch a contiguous byte range into L2 (TMA bulk prefetch; size % 16 == 0).
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- activation staging
// The activation vector is kept in shared memory as K/32 rows of 128 bytes
// (one 32-element block per row) with the 16-byte chunks of row b stored at
// chunk position (m ^ (b & 7)).  A lane reading chunk m of block b and its
// neighbours reading the same chunk of blocks b+1..b+7 then hit eight
// distinct bank groups: 128-bit shared loads are conflict-free.
__device__ __forceinline__ int xswz(int b, int m) { return (b << 3) + (m ^ (b & 7)); }

__device__ __forceinline__ float4 ld_xchunk(const float *xs, int b, int m)
{
    return reinterpret_cast<const float4 *>(xs)[xswz(b, m)];
}

// Copy x[0..K) (16-byte aligned, K % 32 == 0) into the swizzled layout;
// all threads of the CTA take part.  Ends with a CTA barrier.
__device__ __forceinline__ void stage_x(float *xs, const float *__restrict__ x, int K)
{
    const int nchunks = K >> 2;
    for (int c = threadIdx.x; c < nchunks; c += blockDim.x)
        cp_async16(reinterpret_cast<float4 *>(xs) + xswz(c >> 3, c & 7), x + 4 * c);
    cp_async_wait_all();
    __syncthreads();
}

// ---------------------------------------------------------------- reductions
// Sum over aligned groups of LG lanes; every lane of the group gets the sum.
template <int LG>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = LG / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- exact code -> f32
// Four-bit codes are turned into exact f32 values without an int-to-float
// conversion: OR-ing the code (at bit position p < 20) into the bit pattern
// of 2^23 gives the float 2^23 + q * 2^p exactly; one FMA with 2^-p and a
// constant then removes 2^(23-p) (and the Q4_0 offset 8) without rounding,
// since the exact result is a small integer.
constexpr uint32_t kMagic = 0x4B000000u;  // bit pattern of 2^23

__device__ __forceinline__ float2 mk2(float a, float b) { return make_float2(a, b); }

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float2 nib2(uint32_t va, uint32_t ma, uint32_t vb, uint32_t mb)
{
    return make_float2(__uint_as_float((va & ma) | kMagic), __uint_as_float((vb & mb) | kMagic));
}

// q - OFF for the eight nibbles of word w (element order: nibble e of the
// word at bits 4e..4e+3), accumulated against x[0..8) into acc:
//   acc += (q_e - OFF) * x_e, as four packed f32x2 FMAs.
// OFF = 8 for Q4_0 (centred codes), 0 for Q4_K (plain codes).
template <int OFF>
__device__ __forceinline__ float2 nib8_dot(uint32_t w, float4 xa, float4 xb, float2 acc)
{
    constexpr float o = static_cast<float>(OFF);
    const uint32_t v = w, u = w >> 12;  // u holds nibbles 5,6,7 at bits 8,12,16
    // nibbles 0,1 at bits 0,4
    float2 q01 = ffma2(nib2(v, 0xFu, v, 0xF0u), mk2(1.0f, 0x1p-4f),
                       mk2(-(0x1p23f + o), -(0x1p19f + o)));
    // nibbles 2,3 at bits 8,12
    float2 q23 = ffma2(nib2(v, 0xF00u, v, 0xF000u), mk2(0x1p-8f, 0x1p-12f),
                       mk2(-(0x1p15f + o), -(0x1p11f + o)));
    // nibble 4 at bit 16 of v, nibble 5 at bit 8 of u
    float2 q45 = ffma2(nib2(v, 0xF0000u, u, 0xF00u), mk2(0x1p-16f, 0x1p-8f),
                       mk2(-(0x1p7f + o), -(0x1p15f + o)));
    // nibbles 6,7 at bits 12,16 of u
    float2 q67 = ffma2(nib2(u, 0xF000u, u, 0xF0000u), mk2(0x1p-12f, 0x1p-16f),
                       mk2(-(0x1p11f + o), -(0x1p7f + o)));
    acc = ffma2(q01, mk2(xa.x, xa.y), acc);
    acc = ffma2(q23, mk2(xa.z, xa.w), acc);
    acc = ffma2(q45, mk2(xb.x, xb.y), acc);
    acc = ffma2(q67, mk2(xb.z, xb.w), acc);
    return acc;
}

// Offset-binary bytes (u = q + 128) to exact f32 q: PRMT places byte k in
// the low byte of 0x4B0000uu (= 2^23 + u); subtracting 2^23 + 128 is exact.
__device__ __forceinline__ float byte_f(uint32_t w, uint32_t sel)
{
    return __uint_as_float(__byte_perm(w, kMagic, sel));
}
// acc += q * x for the four bytes of w against x4.
__device__ __forceinline__ float2 byte4_dot(uint32_t w, float4 x4, float2 acc)
{
    const float2 off = mk2(-(0x1p23f + 128.0f), -(0x1p23f + 128.0f));
    float2 q01 = __fadd2_rn(mk2(byte_f(w, 0x7540u), byte_f(w, 0x7541u)), off);
    float2 q23 = __fadd2_rn(mk2(byte_f(w, 0x7542u), byte_f(w, 0x7543u)), off);
    acc = ffma2(q01, mk2(x4.x, x4.y), acc);
    acc = ffma2(q23, mk2(x4.z, x4.w), acc);
    return acc;
}

// ---------------------------------------------------------------- top-k keys
// A (value, row) pair as one unsigned 64-bit key whose unsigned order is the
// ranking order: larger value first, equal values by lower row, NaN below
// every number, -0 equal to +0.  Key 0 never occurs for a real row and
// serves as "empty".
__device__ __forceinline__ uint32_t f32_rank(float v)
{
    if (v != v) return 0u;
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ unsigned long long topk_key(float v, uint32_t row)
{
    return (static_cast<unsigned long long>(f32_rank(v)) << 32) | (0xFFFFFFFFu - row);
}
__device__ __forceinline__ float key_value(unsigned long long key)
{
    uint32_t r = static_cast<uint32_t>(key >> 32);
    if (r == 0u) return __uint_as_float(0x7FC00000u);
    return __uint_as_float((r & 0x80000000u) ? (r & 0x7FFFFFFFu) : ~r);
}
__device__ __forceinline__ uint32_t key_row(unsigned long long key)
{
    return 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
}

// A warp-resident sorted list of the k best keys (k <= 64): lane j holds
// entries j (e0) and j + 32 (e1), in descending order.
struct WarpTopK {
    unsigned long long e0, e1;
    __device__ __forceinline__ void init() { e0 = 0ull; e1 = 0ull; }
    // Key of entry k-1 (the admission threshold), same in every lane.
    __device__ __forceinline__ unsigned long long kth(int k) const
    {
        const int i = k - 1;
        unsigned long long v = (i < 32) ? e0 : e1;
        return __shfl_sync(0xffffffffu, v, i & 31);
    }
    // Insert `key` (warp-uniform) keeping the first k entries sorted.
    __device__ __forceinline__ void insert(unsigned long long key, int k)
    {
        const int lane = threadIdx.x & 31;
        const int p = __popc(__ballot_sync(0xffffffffu, e0 > key)) +
                      __popc(__ballot_sync(0xffffffffu, e1 > key));
        if (p >= k) return;
        unsigned long long up0 = __shfl_up_sync(0xffffffffu, e0, 1);
        unsigned long long up1 = __shfl_up_sync(0xffffffffu, e1, 1);
        const unsigned long long last0 = __shfl_sync(0xffffffffu, e0, 31);
        if (lane == 0) up1 = last0;
        const int j0 = lane, j1 = lane + 32;
        e0 = (j0 < p) ? e0 : (j0 == p) ? key : up0;
        e1 = (j1 < p) ? e1 : (j1 == p) ? key : up1;
    }
};

}  // namespace gq
