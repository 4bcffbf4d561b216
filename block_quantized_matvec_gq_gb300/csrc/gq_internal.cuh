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
// hint is accepted by sm_103a only on the 32-byte form.)  The asm is not
// volatile: weights are read-only for the whole kernel, so the compiler may
// schedule these loads like any other load -- a volatile form pinned them in
// program order and cost the 4-bit matvecs a third of their issue rate
// (measured: 7.0 against 10.0 T codes/s per GPU on the same core).
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
// 32-byte load (two 16-byte halves), evict-first in L2.
__device__ __forceinline__ void ld_stream32(const void *p, uint4 &a, uint4 &b)
{
    asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
        : "l"(p));
}
__device__ __forceinline__ uint16_t ld_stream_u16(const void *p)
{
    uint16_t v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
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
// Codes are turned into exact f32 values without an int-to-float
// conversion: OR-ing a code into the significand of a power of two 2^e, with
// the code's lowest bit on the units place (bit 23 - e of the significand),
// gives the float 2^e + q exactly; one add of -(2^e + offset) then leaves
// (q - offset) without rounding, since the exact result is a small integer.
constexpr uint32_t kMagic = 0x4B000000u;  // bit pattern of 2^23

__device__ __forceinline__ float2 mk2(float a, float b) { return make_float2(a, b); }

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ---------------------------------------------------------------- 4-bit codes
// One 32-bit word w holds the 8 nibbles of one 8-element group in element
// order (nibble k = bits 4k..4k+3).  For i = 0..3 the pair (nibble i, nibble
// i+4) is isolated in place by one LOP3 each into an f32 whose exponent is
// chosen per pair: OR-ing (w & 0xF<<4i) into the bit pattern of 2^(23-4i)
// puts the nibble on the units bit of the significand, so the float is
// exactly 2^(23-4i) + q (and the same on w>>16 gives element i+4).  One
// packed f32x2 add of -(2^(23-4i) + OFF) turns the pair into
// (q_i - OFF, q_{i+4} - OFF) exactly, and one packed FMA adds its products
// with (x_i, x_{i+4}).  x is staged per 8-group in the order
// x0,x4,x1,x5,x2,x6,x3,x7, so each pair of x values is one aligned 64-bit
// register pair.  The whole word is one asm block so that the LOP3 results
// land directly in the 64-bit pairs the packed instructions read.
#define GQ_NIB8_BODY(FIRST)                                                                                      \
    "{\n"                                                                                                        \
    " .reg .b32 h, l0, h0, l1, h1, l2, h2, l3, h3;\n"                                                           \
    " .reg .b64 p0, p1, p2, p3, x0, x1, x2, x3, a, c0, c1, c2, c3;\n"                                           \
    " shr.u32 h, %2, 16;\n"                                                                                      \
    " lop3.b32 l0, %2, 0x0000000F, 0x4B000000, 0xEA;\n lop3.b32 h0, h, 0x0000000F, 0x4B000000, 0xEA;\n"         \
    " lop3.b32 l1, %2, 0x000000F0, 0x49000000, 0xEA;\n lop3.b32 h1, h, 0x000000F0, 0x49000000, 0xEA;\n"         \
    " lop3.b32 l2, %2, 0x00000F00, 0x47000000, 0xEA;\n lop3.b32 h2, h, 0x00000F00, 0x47000000, 0xEA;\n"         \
    " lop3.b32 l3, %2, 0x0000F000, 0x45000000, 0xEA;\n lop3.b32 h3, h, 0x0000F000, 0x45000000, 0xEA;\n"         \
    " mov.b64 p0, {l0, h0};\n mov.b64 p1, {l1, h1};\n mov.b64 p2, {l2, h2};\n mov.b64 p3, {l3, h3};\n"         \
    " mov.b64 c0, {%13, %13};\n mov.b64 c1, {%14, %14};\n mov.b64 c2, {%15, %15};\n mov.b64 c3, {%16, %16};\n" \
    " add.rn.f32x2 p0, p0, c0;\n add.rn.f32x2 p1, p1, c1;\n add.rn.f32x2 p2, p2, c2;\n add.rn.f32x2 p3, p3, c3;\n"  \
    " mov.b64 x0, {%3, %4};\n mov.b64 x1, {%5, %6};\n mov.b64 x2, {%7, %8};\n mov.b64 x3, {%9, %10};\n"         \
    " mov.b64 a, {%11, %12};\n" FIRST                                                                            \
    " fma.rn.f32x2 a, p1, x1, a;\n fma.rn.f32x2 a, p2, x2, a;\n fma.rn.f32x2 a, p3, x3, a;\n"                   \
    " mov.b64 {%0, %1}, a;\n"                                                                                    \
    "}"

// -(2^(23-4i) + OFF): removes pair i's exponent term and the code offset.
template <int OFF>
struct NibConsts {
    static constexpr float c0 = -(8388608.0f + OFF);  // -(2^23 + OFF)
    static constexpr float c1 = -(524288.0f + OFF);   // -(2^19 + OFF)
    static constexpr float c2 = -(32768.0f + OFF);    // -(2^15 + OFF)
    static constexpr float c3 = -(2048.0f + OFF);     // -(2^11 + OFF)
};

// Returns acc + sum over the word of (q - OFF) * x as a packed pair of
// partial sums; kStart ignores acc (starts a new chain).
template <int OFF, bool kStart>
__device__ __forceinline__ float2 nib8_fma(uint32_t w, float4 xa, float4 xb, float2 acc)
{
    float2 r;
    if (kStart) {
        asm(GQ_NIB8_BODY(" mul.rn.f32x2 a, p0, x0;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y), "f"(xb.z), "f"(xb.w),
              "f"(acc.x), "f"(acc.y), "f"(NibConsts<OFF>::c0), "f"(NibConsts<OFF>::c1), "f"(NibConsts<OFF>::c2),
              "f"(NibConsts<OFF>::c3));
    } else {
        asm(GQ_NIB8_BODY(" fma.rn.f32x2 a, p0, x0, a;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y), "f"(xb.z), "f"(xb.w),
              "f"(acc.x), "f"(acc.y), "f"(NibConsts<OFF>::c0), "f"(NibConsts<OFF>::c1), "f"(NibConsts<OFF>::c2),
              "f"(NibConsts<OFF>::c3));
    }
    return r;
}

// ---------------------------------------------------------------- offset-free 4-bit codes as subnormals
// A code without offset (Q4_K: w = d*sc*q - dmin*m) need not be converted at
// all: AND-ing nibble i (bits 4i..4i+3) out of a 16-bit half leaves, with a
// zero exponent field, the bit pattern of the subnormal f32 q * 2^(4i-149).
// If the staged x of that position holds x * 2^(149-4i-c) (stage_x_q4k), the
// FMA forms q * x * 2^-c from the exact product and rounds once, as the
// magic-number form does with (q - OFF) * x; the sum comes out scaled by
// 2^-c.  Per 8 codes: one shift, eight ANDs and four packed FMAs, against
// eight LOP3s, four packed adds and four packed FMAs.  Subnormal operands
// are kept: the PTX operations carry no .ftz.
#define GQ_NIB8_SUB_BODY(FIRST)                                                              \
    "{\n"                                                                                    \
    " .reg .b32 h, l0, h0, l1, h1, l2, h2, l3, h3;\n"                                       \
    " .reg .b64 p0, p1, p2, p3, x0, x1, x2, x3, a;\n"                                       \
    " shr.u32 h, %2, 16;\n"                                                                  \
    " and.b32 l0, %2, 0x0000000F;\n and.b32 h0, h, 0x0000000F;\n"                           \
    " and.b32 l1, %2, 0x000000F0;\n and.b32 h1, h, 0x000000F0;\n"                           \
    " and.b32 l2, %2, 0x00000F00;\n and.b32 h2, h, 0x00000F00;\n"                           \
    " and.b32 l3, %2, 0x0000F000;\n and.b32 h3, h, 0x0000F000;\n"                           \
    " mov.b64 p0, {l0, h0};\n mov.b64 p1, {l1, h1};\n mov.b64 p2, {l2, h2};\n mov.b64 p3, {l3, h3};\n" \
    " mov.b64 x0, {%3, %4};\n mov.b64 x1, {%5, %6};\n mov.b64 x2, {%7, %8};\n mov.b64 x3, {%9, %10};\n" \
    " mov.b64 a, {%11, %12};\n" FIRST                                                        \
    " fma.rn.f32x2 a, p1, x1, a;\n fma.rn.f32x2 a, p2, x2, a;\n fma.rn.f32x2 a, p3, x3, a;\n" \
    " mov.b64 {%0, %1}, a;\n"                                                                \
    "}"

// Returns acc + sum over the word of q * xs (xs the position-scaled staged
// x) as a packed pair of partial sums; kStart ignores acc.
template <bool kStart>
__device__ __forceinline__ float2 nib8_sub_fma(uint32_t w, float4 xa, float4 xb, float2 acc)
{
    float2 r;
    if (kStart) {
        asm(GQ_NIB8_SUB_BODY(" mul.rn.f32x2 a, p0, x0;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y), "f"(xb.z), "f"(xb.w),
              "f"(acc.x), "f"(acc.y));
    } else {
        asm(GQ_NIB8_SUB_BODY(" fma.rn.f32x2 a, p0, x0, a;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y), "f"(xb.z), "f"(xb.w),
              "f"(acc.x), "f"(acc.y));
    }
    return r;
}

// 2^k as f32 for -126 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }
// v * 2^k for -252 <= k <= 254 in two exact power-of-two steps.
__device__ __forceinline__ float scale_pow2(float v, int k)
{
    const int k1 = k >> 1;
    return v * pow2i(k1) * pow2i(k - k1);
}

// ---------------------------------------------------------------- activation staging for 4-bit formats
// x is kept in shared memory as K/32 blocks of kXBlk = 36 floats (144 bytes):
// the block's 32 values, every 8-element group in the order
// 0,4,1,5,2,6,3,7 (the pair order of nib8_fma), then the block's sum of x
// (the Q4_K min term) and 3 unused floats.  Lanes reading the same 16-byte
// chunk of consecutive blocks are 144 bytes apart, i.e. on distinct bank
// groups, so 128-bit loads are conflict-free with a fixed immediate offset
// per chunk.
constexpr int kXBlk = 36;

__device__ __forceinline__ float4 ld_xq4(const float *xb, int m)
{
    return *reinterpret_cast<const float4 *>(xb + 4 * m);
}

// All threads of the CTA take part; ends with a CTA barrier.
// A long vector (more than two 8-groups per thread) has four 8-groups per
// thread loaded before any is stored, so it waits for L2 about once per four
// groups rather than once per group; a short one keeps the plain loop (the
// 4096-element vector measured 0.2 us slower with the unrolled form).
template <bool kWithSum>
__device__ __forceinline__ void stage_x_q4(float *xs, const float *__restrict__ x, int K)
{
    const int ngroups = K >> 3;
    constexpr int kB = 4;
    if (ngroups <= 2 * static_cast<int>(blockDim.x)) {
        for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
            const float4 a = *reinterpret_cast<const float4 *>(x + 8 * g);
            const float4 b = *reinterpret_cast<const float4 *>(x + 8 * g + 4);
            float *dst = xs + (g >> 2) * kXBlk + 8 * (g & 3);
            *reinterpret_cast<float4 *>(dst) = make_float4(a.x, b.x, a.y, b.y);
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(a.z, b.z, a.w, b.w);
        }
    } else {
        for (int g0 = threadIdx.x; g0 < ngroups; g0 += kB * blockDim.x) {
            float4 a[kB], b[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const int g = g0 + j * static_cast<int>(blockDim.x);
                if (g < ngroups) {
                    a[j] = *reinterpret_cast<const float4 *>(x + 8 * g);
                    b[j] = *reinterpret_cast<const float4 *>(x + 8 * g + 4);
                }
            }
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const int g = g0 + j * static_cast<int>(blockDim.x);
                if (g < ngroups) {
                    float *dst = xs + (g >> 2) * kXBlk + 8 * (g & 3);
                    *reinterpret_cast<float4 *>(dst) = make_float4(a[j].x, b[j].x, a[j].y, b[j].y);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(a[j].z, b[j].z, a[j].w, b[j].w);
                }
            }
        }
    }
    if (kWithSum) {
        __syncthreads();
        for (int b = threadIdx.x; b < (K >> 5); b += blockDim.x) {
            const float *src = xs + b * kXBlk;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 v = ld_xq4(src, m);
                s += v.x;
                s += v.y;
                s += v.z;
                s += v.w;
            }
            xs[b * kXBlk + 32] = s;
        }
    }
    __syncthreads();
}

// Bit pattern of |v| if v is finite, else 0 (the unsigned order of these
// patterns is the order of the magnitudes).
__device__ __forceinline__ uint32_t finite_mag_bits(float v)
{
    const uint32_t b = __float_as_uint(v) & 0x7FFFFFFFu;
    return b < 0x7F800000u ? b : 0u;
}

// Staging for the subnormal-code core (nib8_sub_fma): the layout of
// stage_x_q4<true>, with every value multiplied by 2^(149-4i-c), i its
// nibble position (stored index t of an 8-group has i = t/2), and the block
// sums (taken from the unscaled values: each lane sums its 8-group in stored
// order, then the four lanes of the block add theirs with two butterfly
// shuffles) by 2^-c.  c = e + 22, e the binary exponent of the largest finite
// |x| (at least -126): the largest scaled value stays below 2^128, and a
// product q * x * 2^-c is a normal number whenever |x| >= 2^(e-104).
// Infinities and NaNs stay what they are.  K % 32 == 0.  Returns c (the same
// in every thread); all threads of the CTA take part (blockDim.x a multiple
// of 32); `red` holds one word per warp; ends with a CTA barrier.
__device__ __forceinline__ int stage_x_q4k(float *xs, const float *__restrict__ x, int K, uint32_t *red)
{
    const int ngroups = K >> 3;  // a multiple of 4: the 4 groups of a block sit on 4 adjacent lanes
    uint32_t mx = 0u;
    for (int g0 = threadIdx.x & ~31; g0 < ngroups; g0 += blockDim.x) {
        const int g = g0 + (threadIdx.x & 31);
        float s = 0.f;
        if (g < ngroups) {
            const float4 a = *reinterpret_cast<const float4 *>(x + 8 * g);
            const float4 b = *reinterpret_cast<const float4 *>(x + 8 * g + 4);
            float *dst = xs + (g >> 2) * kXBlk + 8 * (g & 3);
            *reinterpret_cast<float4 *>(dst) = make_float4(a.x, b.x, a.y, b.y);
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(a.z, b.z, a.w, b.w);
            mx = max(mx, max(max(finite_mag_bits(a.x), finite_mag_bits(a.y)), max(finite_mag_bits(a.z), finite_mag_bits(a.w))));
            mx = max(mx, max(max(finite_mag_bits(b.x), finite_mag_bits(b.y)), max(finite_mag_bits(b.z), finite_mag_bits(b.w))));
            s = a.x;
            s += b.x;
            s += a.y;
            s += b.y;
            s += a.z;
            s += b.z;
            s += a.w;
            s += b.w;
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (g < ngroups && (g & 3) == 0) xs[(g >> 2) * kXBlk + 32] = s;
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) mx = max(mx, red[w]);
    const int e = max(static_cast<int>(mx >> 23) - 127, -126);
    const int c = e + 22;
    // position i's factor 2^(127-e-4i) as two exact powers of two
    float f1[4], f2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = 127 - e - 4 * i, k1 = k >> 1;
        f1[i] = pow2i(k1);
        f2[i] = pow2i(k - k1);
    }
    const int ks = -c, ks1 = ks >> 1;
    const float s1 = pow2i(ks1), s2 = pow2i(ks - ks1);
    for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
        float *p = xs + (g >> 2) * kXBlk + 8 * (g & 3);
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        *reinterpret_cast<float4 *>(p) =
            make_float4(a.x * f1[0] * f2[0], a.y * f1[0] * f2[0], a.z * f1[1] * f2[1], a.w * f1[1] * f2[1]);
        *reinterpret_cast<float4 *>(p + 4) =
            make_float4(b.x * f1[2] * f2[2], b.y * f1[2] * f2[2], b.z * f1[3] * f2[3], b.w * f1[3] * f2[3]);
        if ((g & 3) == 0) p[32] = p[32] * s1 * s2;
    }
    __syncthreads();
    return c;
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
// Sort 128 keys held 4 per lane (key i = lane + 32*j in e[j]) into
// descending order with a bitonic network: strides 64 and 32 exchange within
// a lane, smaller strides between lanes.  28 parallel compare-exchange
// stages.
__device__ __forceinline__ void warp_sort128_desc(unsigned long long (&e)[4])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 128; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32) {
                const int js = stride >> 5;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if ((j & js) == 0) {
                        const int i = lane + 32 * j;
                        const bool desc = (i & size) == 0;  // this block of `size` sorts descending
                        const unsigned long long a = e[j], b = e[j | js];
                        const bool swap = desc ? (a < b) : (a > b);
                        e[j] = swap ? b : a;
                        e[j | js] = swap ? a : b;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = lane + 32 * j;
                    const bool desc = (i & size) == 0;
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, e[j], stride);
                    const bool lower = (lane & stride) == 0;  // this key is the lower index of the pair
                    // lower index keeps the larger key when the block is descending
                    const bool keep_max = (lower == desc);
                    e[j] = keep_max ? (e[j] > other ? e[j] : other) : (e[j] < other ? e[j] : other);
                }
            }
        }
    }
}

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
