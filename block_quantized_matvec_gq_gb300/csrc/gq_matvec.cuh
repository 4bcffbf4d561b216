// gq_matvec.cuh -- weight-streaming cores of the decode matvecs.
//
// Geometry (all compile-time): a warp is split into G = 32/LG lane groups of
// LG lanes; each lane group owns NS row streams at a time, and lane lp of a
// group handles blocks lp, lp+LG, lp+2LG, ... of each of its rows.  One x
// block (32 floats, from the swizzled shared copy) is loaded once per lane
// and used for all NS rows; lanes of different groups that read the same x
// block get a shared-memory broadcast.  Per row and lane the products are
// summed per block in packed f32x2 registers, scaled by the block's d, and
// accumulated across the lane's blocks; the group then reduces its LG
// partial sums with shuffles.  U blocks per row are loaded before any is
// used, so each lane keeps U*NS 16-byte weight loads in flight.
#pragma once

#include "gq_internal.cuh"

namespace gq {

// ---------------------------------------------------------------- Q4_0
// Packed Q4_0: nibble plane (16 B per block, element order) + fp16 scale plane.
template <int LG, int NS, int U>
__device__ __forceinline__ void q4_0_stream(const uint4 *const (&wp)[NS],
                                            const uint16_t *const (&sp)[NS], const float *xs,
                                            int nb, int lp, float (&out)[NS])
{
    float2 acc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);

    for (int b0 = lp; b0 < nb; b0 += LG * U) {
        uint4 w[U][NS];
        float d[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            const bool ok = b < nb;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                w[u][i] = ok ? ld_stream16(wp[i] + b) : make_uint4(0u, 0u, 0u, 0u);
                d[u][i] = ok ? __half2float(__ushort_as_half(ld_stream_u16(sp[i] + b))) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            if (b < nb) {
                float4 xv[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) xv[m] = ld_xchunk(xs, b, m);
                float2 blk[NS];
#pragma unroll
                for (int i = 0; i < NS; ++i) blk[i] = nib32_dot_h<8>(w[u][i], xv);
#pragma unroll
                for (int i = 0; i < NS; ++i) acc[i] = ffma2(blk[i], make_float2(d[u][i], d[u][i]), acc[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
}

// ---------------------------------------------------------------- Q8_0
// Packed Q8_0: byte plane (32 B per block, offset binary) + fp16 scale plane.
template <int LG, int NS, int U>
__device__ __forceinline__ void q8_0_stream(const uint4 *const (&wp)[NS],
                                            const uint16_t *const (&sp)[NS], const float *xs,
                                            int nb, int lp, float (&out)[NS])
{
    float2 acc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);

    for (int b0 = lp; b0 < nb; b0 += LG * U) {
        uint4 w[U][NS][2];
        float d[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            const bool ok = b < nb;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                if (ok) {
                    ld_stream32(wp[i] + 2 * b, w[u][i][0], w[u][i][1]);
                } else {
                    w[u][i][0] = make_uint4(0u, 0u, 0u, 0u);
                    w[u][i][1] = make_uint4(0u, 0u, 0u, 0u);
                }
                d[u][i] = ok ? __half2float(__ushort_as_half(ld_stream_u16(sp[i] + b))) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            if (b < nb) {
                float4 xv[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) xv[m] = ld_xchunk(xs, b, m);
                float2 blk[NS];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const uint4 &h0 = w[u][i][0];
                    const uint4 &h1 = w[u][i][1];
                    const float2 p0 = byte4_dot(h0.y, xv[1], byte4_part(h0.x, xv[0]));
                    const float2 p1 = byte4_dot(h0.w, xv[3], byte4_part(h0.z, xv[2]));
                    const float2 p2 = byte4_dot(h1.y, xv[5], byte4_part(h1.x, xv[4]));
                    const float2 p3 = byte4_dot(h1.w, xv[7], byte4_part(h1.z, xv[6]));
                    blk[i] = __fadd2_rn(__fadd2_rn(p0, p1), __fadd2_rn(p2, p3));
                }
#pragma unroll
                for (int i = 0; i < NS; ++i) acc[i] = ffma2(blk[i], make_float2(d[u][i], d[u][i]), acc[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
}

// ---------------------------------------------------------------- Q4_K
// Packed Q4_K: nibble plane (128 B per super-block, sub-block s at 16 s, element
// order) + record plane (16 B per super-block: d, dmin, 12 scale bytes).
// A lane handles one 32-weight sub-block per step: sub-block index sb (global
// within the row), super-block sb/8, sub-block s = sb%8.  xsum holds the sum
// of each 32-element block of x (shared memory).
__device__ __forceinline__ void q4k_scale_min(uint4 rec, int s, float &sc, float &mn)
{
    const int sh = 8 * (s & 3);
    const uint32_t A = (rec.y >> sh) & 0xFFu;  // scale byte s&3
    const uint32_t B = (rec.z >> sh) & 0xFFu;  // scale byte (s&3)+4
    const uint32_t C = (rec.w >> sh) & 0xFFu;  // scale byte (s&3)+8
    uint32_t isc, imn;
    if (s < 4) {
        isc = A & 63u;
        imn = B & 63u;
    } else {
        isc = (C & 15u) | ((A >> 6) << 4);
        imn = (C >> 4) | ((B >> 6) << 4);
    }
    sc = static_cast<float>(isc);
    mn = static_cast<float>(imn);
}

template <int LG, int NS, int U>
__device__ __forceinline__ void q4k_stream(const uint4 *const (&wp)[NS], const uint4 *const (&rp)[NS],
                                           const float *xs, const float *xsum, int nsb, int lp,
                                           float (&out)[NS])
{
    float2 acc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);

    for (int b0 = lp; b0 < nsb; b0 += LG * U) {
        uint4 w[U][NS];
        uint4 rec[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            const bool ok = b < nsb;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                w[u][i] = ok ? ld_stream16(wp[i] + b) : make_uint4(0u, 0u, 0u, 0u);
                // the 16-byte record is shared by the 8 lanes of a super-block
                rec[u][i] = ok ? __ldg(rp[i] + (b >> 3)) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + u * LG;
            if (b < nsb) {
                float4 xv[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) xv[m] = ld_xchunk(xs, b, m);
                float2 blk[NS];
#pragma unroll
                for (int i = 0; i < NS; ++i) blk[i] = nib32_dot_h<0>(w[u][i], xv);
                const float xsb = xsum[b];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    float sc, mn;
                    q4k_scale_min(rec[u][i], b & 7, sc, mn);
                    const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(rec[u][i].x & 0xFFFFu)));
                    const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(rec[u][i].x >> 16)));
                    // d*sc and dmin*m are exact in f32 (11-bit x 6-bit products)
                    const float dsc = d * sc, dm = dmin * mn;
                    acc[i].x = fmaf(dsc, blk[i].x, acc[i].x);
                    acc[i].y = fmaf(dsc, blk[i].y, acc[i].y);
                    acc[i].x = fmaf(-dm, xsb, acc[i].x);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
}


// ---------------------------------------------------------------- 32-byte loads (block pairs)
// Same arithmetic with two consecutive blocks per lane and row per load (one
// 256-bit load of 32 nibble bytes, one 32-bit load of the two scales): twice
// the bytes per memory request of the one-block form.  Lane lp of a group
// takes pairs lp, lp+LG, ...; pair p is blocks 2p and 2p+1 (nb even).
__device__ __forceinline__ uint32_t ld_stream_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <int LG, int NS, int U>
__device__ __forceinline__ void q4_0_stream2(const uint4 *const (&wp)[NS], const uint16_t *const (&sp)[NS],
                                             const float *xs, int nb, int lp, float (&out)[NS])
{
    const int np = nb >> 1;
    float2 acc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);

    for (int p0 = lp; p0 < np; p0 += LG * U) {
        uint4 w[U][NS][2];
        uint32_t dd[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u * LG;
            const bool ok = p < np;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                if (ok) {
                    ld_stream32(wp[i] + 2 * p, w[u][i][0], w[u][i][1]);
                    dd[u][i] = ld_stream_u32(sp[i] + 2 * p);
                } else {
                    w[u][i][0] = make_uint4(0u, 0u, 0u, 0u);
                    w[u][i][1] = make_uint4(0u, 0u, 0u, 0u);
                    dd[u][i] = 0u;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u * LG;
            if (p < np) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = 2 * p + h;
                    float4 xv[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) xv[m] = ld_xchunk(xs, b, m);
                    float2 blk[NS];
#pragma unroll
                    for (int i = 0; i < NS; ++i) blk[i] = nib32_dot_h<8>(w[u][i][h], xv);
#pragma unroll
                    for (int i = 0; i < NS; ++i) {
                        const uint16_t hb = static_cast<uint16_t>(h ? (dd[u][i] >> 16) : (dd[u][i] & 0xFFFFu));
                        const float d = __half2float(__ushort_as_half(hb));
                        acc[i] = ffma2(blk[i], make_float2(d, d), acc[i]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
}

template <int LG, int NS, int U>
__device__ __forceinline__ void q4k_stream2(const uint4 *const (&wp)[NS], const uint4 *const (&rp)[NS],
                                            const float *xs, const float *xsum, int nsb, int lp, float (&out)[NS])
{
    const int np = nsb >> 1;
    float2 acc[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);

    for (int p0 = lp; p0 < np; p0 += LG * U) {
        uint4 w[U][NS][2];
        uint4 rec[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u * LG;
            const bool ok = p < np;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                if (ok) {
                    ld_stream32(wp[i] + 2 * p, w[u][i][0], w[u][i][1]);
                    rec[u][i] = __ldg(rp[i] + (p >> 2));  // both sub-blocks lie in super-block p/4
                } else {
                    w[u][i][0] = make_uint4(0u, 0u, 0u, 0u);
                    w[u][i][1] = make_uint4(0u, 0u, 0u, 0u);
                    rec[u][i] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u * LG;
            if (p < np) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = 2 * p + h;
                    float4 xv[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) xv[m] = ld_xchunk(xs, b, m);
                    float2 blk[NS];
#pragma unroll
                    for (int i = 0; i < NS; ++i) blk[i] = nib32_dot_h<0>(w[u][i][h], xv);
                    const float xsb = xsum[b];
#pragma unroll
                    for (int i = 0; i < NS; ++i) {
                        float sc, mn;
                        q4k_scale_min(rec[u][i], b & 7, sc, mn);
                        const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(rec[u][i].x & 0xFFFFu)));
                        const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(rec[u][i].x >> 16)));
                        const float dsc = d * sc, dm = dmin * mn;
                        acc[i].x = fmaf(dsc, blk[i].x, acc[i].x);
                        acc[i].y = fmaf(dsc, blk[i].y, acc[i].y);
                        acc[i].x = fmaf(-dm, xsb, acc[i].x);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
}

// ---------------------------------------------------------------- kernel-side common
constexpr int kThreadsPerCta = 256;
constexpr int kWarpsPerCta = kThreadsPerCta / 32;

// Before waiting on the previous kernel, ask L2 to fetch the weight rows of
// this warp's first task (weights never depend on the previous kernel).
// One lane per row issues a bulk prefetch of the whole row.
template <int NS>
__device__ __forceinline__ void prefetch_rows_l2(const void *const (&rowp)[NS], uint32_t row_bytes, int lane)
{
#pragma unroll
    for (int i = 0; i < NS; ++i)
        if (lane == i) prefetch_l2_bulk(rowp[i], row_bytes);
}

// Per-block sums of x (for the min term), after stage_x.
__device__ __forceinline__ void stage_xsum(float *xsum, const float *xs, int nb)
{
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float4 v = ld_xchunk(xs, b, m);
            s += v.x;
            s += v.y;
            s += v.z;
            s += v.w;
        }
        xsum[b] = s;
    }
    __syncthreads();
}

// GELU, tanh form, with the tanh argument clamped to +-15 (tanh(15) rounds
// to 1 in f32, so the clamp changes no finite result and keeps it finite).
__device__ __forceinline__ float gelu_tanh(float a)
{
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    float t = k0 * (a + 0.044715f * a * a * a);
    t = fminf(fmaxf(t, -15.f), 15.f);
    return 0.5f * a * (1.f + tanhf(t));
}

}  // namespace gq

// ---------------------------------------------------------------- host-side dispatch
// Every matvec-family kernel is instantiated for these geometries; the
// entry points pick one by shape (choose_matvec_geo).
#define GQ_GEO_CASE1(geo, CASE, LG, R)                                  \
    if ((geo).lg == LG && (geo).r == R && (geo).u == 2) { CASE(LG, R, 2); } \
    if ((geo).lg == LG && (geo).r == R && (geo).u == 4) { CASE(LG, R, 4); }
#define GQ_GEO_SWITCH(geo, CASE)              \
    do {                                      \
        GQ_GEO_CASE1(geo, CASE, 32, 1)        \
        GQ_GEO_CASE1(geo, CASE, 32, 2)        \
        GQ_GEO_CASE1(geo, CASE, 32, 4)        \
        GQ_GEO_CASE1(geo, CASE, 16, 1)        \
        GQ_GEO_CASE1(geo, CASE, 16, 2)        \
        GQ_GEO_CASE1(geo, CASE, 16, 4)        \
        GQ_GEO_CASE1(geo, CASE, 8, 1)         \
        GQ_GEO_CASE1(geo, CASE, 8, 2)         \
        GQ_GEO_CASE1(geo, CASE, 8, 4)         \
        return GQ_ERR_SHAPE;                  \
    } while (0)
// Block-pair (32-byte load) kernels: LG in {4, 8, 16, 32}, R in {1, 2}, U in {2, 4}.
#define GQ_PAIR_SWITCH(geo, CASE)             \
    do {                                      \
        GQ_GEO_CASE1(geo, CASE, 32, 1)        \
        GQ_GEO_CASE1(geo, CASE, 32, 2)        \
        GQ_GEO_CASE1(geo, CASE, 16, 1)        \
        GQ_GEO_CASE1(geo, CASE, 16, 2)        \
        GQ_GEO_CASE1(geo, CASE, 8, 1)         \
        GQ_GEO_CASE1(geo, CASE, 8, 2)         \
        GQ_GEO_CASE1(geo, CASE, 4, 1)         \
        GQ_GEO_CASE1(geo, CASE, 4, 2)         \
        return GQ_ERR_SHAPE;                  \
    } while (0)
#define GQ_GEO_SWITCH_R12(geo, CASE)          \
    do {                                      \
        GQ_GEO_CASE1(geo, CASE, 32, 1)        \
        GQ_GEO_CASE1(geo, CASE, 32, 2)        \
        GQ_GEO_CASE1(geo, CASE, 16, 1)        \
        GQ_GEO_CASE1(geo, CASE, 16, 2)        \
        GQ_GEO_CASE1(geo, CASE, 8, 1)         \
        GQ_GEO_CASE1(geo, CASE, 8, 2)         \
        return GQ_ERR_SHAPE;                  \
    } while (0)
