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


// ---------------------------------------------------------------- 4-bit codes via f16 magic
// A second exact route from nibbles to f32 that spends one logic operation
// per TWO codes: OR-ing two nibbles (at bits p and p+16, p < 10) into the
// pattern 0x6400 of each half gives the halves 1024 + q * 2^p exactly; a
// mixed-precision add / fma (f16 source, f32 result and constant) then
// removes 1024 (and the offset) without rounding.  Inside each 8-element
// group the codes come out in the order 0,4,1,5,2,6,3,7, so x is staged in
// that order (stage_x_perm8) and the packed f32x2 FMAs pair them directly.
__device__ __forceinline__ float2 h2_to_f2_add(uint32_t h, float c)
{
    float a, b;
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.f16 %0, lo, %3;\n add.rn.f32.f16 %1, hi, %3;\n}"
        : "=f"(a), "=f"(b)
        : "r"(h), "f"(c));
    return make_float2(a, b);
}
__device__ __forceinline__ float2 h2_to_f2_fma(uint32_t h, uint16_t s, float c)
{
    float a, b;
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %2;\n fma.rn.f32.f16 %0, lo, %3, %4;\n fma.rn.f32.f16 %1, hi, %3, %4;\n}"
        : "=f"(a), "=f"(b)
        : "r"(h), "h"(s), "f"(c));
    return make_float2(a, b);
}
// acc += (q - OFF) . x over the 8 nibbles of w (element order), with x given
// in group order: xa = (x0, x4, x1, x5), xb = (x2, x6, x3, x7).
template <int OFF>
__device__ __forceinline__ float2 nib8_dot_h(uint32_t w, float4 xa, float4 xb, float2 acc)
{
    constexpr float c0 = -(1024.0f + OFF);
    constexpr float c1 = -(64.0f + OFF);
    constexpr uint16_t k16 = 0x2C00;  // f16 1/16
    const uint32_t w2 = w >> 8;
    const float2 q04 = h2_to_f2_add((w & 0x000F000Fu) | 0x64006400u, c0);          // e0, e4
    const float2 q15 = h2_to_f2_fma((w & 0x00F000F0u) | 0x64006400u, k16, c1);     // e1, e5
    const float2 q26 = h2_to_f2_add((w2 & 0x000F000Fu) | 0x64006400u, c0);         // e2, e6
    const float2 q37 = h2_to_f2_fma((w2 & 0x00F000F0u) | 0x64006400u, k16, c1);    // e3, e7
    acc = ffma2(q04, mk2(xa.x, xa.y), acc);
    acc = ffma2(q15, mk2(xa.z, xa.w), acc);
    acc = ffma2(q26, mk2(xb.x, xb.y), acc);
    acc = ffma2(q37, mk2(xb.z, xb.w), acc);
    return acc;
}

// Partial sum of one 32-bit word, started fresh (no incoming accumulator),
// so the words of a block form independent dependency chains that the
// caller adds as a tree.
template <int OFF>
__device__ __forceinline__ float2 nib8_part_h(uint32_t w, float4 xa, float4 xb)
{
    constexpr float c0 = -(1024.0f + OFF);
    constexpr float c1 = -(64.0f + OFF);
    constexpr uint16_t k16 = 0x2C00;  // f16 1/16
    const uint32_t w2 = w >> 8;
    const float2 q04 = h2_to_f2_add((w & 0x000F000Fu) | 0x64006400u, c0);
    const float2 q15 = h2_to_f2_fma((w & 0x00F000F0u) | 0x64006400u, k16, c1);
    const float2 q26 = h2_to_f2_add((w2 & 0x000F000Fu) | 0x64006400u, c0);
    const float2 q37 = h2_to_f2_fma((w2 & 0x00F000F0u) | 0x64006400u, k16, c1);
    float2 acc = __fmul2_rn(q04, mk2(xa.x, xa.y));
    acc = ffma2(q15, mk2(xa.z, xa.w), acc);
    acc = ffma2(q26, mk2(xb.x, xb.y), acc);
    acc = ffma2(q37, mk2(xb.z, xb.w), acc);
    return acc;
}
// Sum over a 16-byte chunk (4 words = 32 nibbles) of one block: four
// independent word chains, added pairwise.
template <int OFF>
__device__ __forceinline__ float2 nib32_dot_h(uint4 w, const float4 (&x)[8])
{
    const float2 a0 = nib8_part_h<OFF>(w.x, x[0], x[1]);
    const float2 a1 = nib8_part_h<OFF>(w.y, x[2], x[3]);
    const float2 a2 = nib8_part_h<OFF>(w.z, x[4], x[5]);
    const float2 a3 = nib8_part_h<OFF>(w.w, x[6], x[7]);
    return __fadd2_rn(__fadd2_rn(a0, a1), __fadd2_rn(a2, a3));
}

// Stage x like stage_x, with every 8-element group stored in the order
// 0,4,1,5,2,6,3,7.  Ends with a CTA barrier.
__device__ __forceinline__ void stage_x_perm8(float *xs, const float *__restrict__ x, int K)
{
    const int ngroups = K >> 3;
    for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
        const float4 a = *reinterpret_cast<const float4 *>(x + 8 * g);
        const float4 b = *reinterpret_cast<const float4 *>(x + 8 * g + 4);
        const int blk = g >> 2, t = g & 3;
        reinterpret_cast<float4 *>(xs)[xswz(blk, 2 * t)] = make_float4(a.x, b.x, a.y, b.y);
        reinterpret_cast<float4 *>(xs)[xswz(blk, 2 * t + 1)] = make_float4(a.z, b.z, a.w, b.w);
    }
    __syncthreads();
}

// Offset-binary bytes (u = q + 128) to exact f32 q: PRMT places byte k in
// the low byte of 0x4B0000uu (= 2^23 + u); subtracting 2^23 + 128 is exact.
__device__ __forceinline__ float byte_f(uint32_t w, uint32_t sel)
{
    return __uint_as_float(__byte_perm(w, kMagic, sel));
}
// q * x for the four bytes of w against x4, started fresh.
__device__ __forceinline__ float2 byte4_part(uint32_t w, float4 x4)
{
    const float2 off = mk2(-(0x1p23f + 128.0f), -(0x1p23f + 128.0f));
    float2 q01 = __fadd2_rn(mk2(byte_f(w, 0x7540u), byte_f(w, 0x7541u)), off);
    float2 q23 = __fadd2_rn(mk2(byte_f(w, 0x7542u), byte_f(w, 0x7543u)), off);
    return ffma2(q23, mk2(x4.z, x4.w), __fmul2_rn(q01, mk2(x4.x, x4.y)));
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
