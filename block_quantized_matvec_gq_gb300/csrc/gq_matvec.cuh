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

// ---------------------------------------------------------------- Q4_0 / Q4_K block core
// Dot products of one 32-weight block (four 32-bit nibble words in element
// order) of NS rows against the block's staged x: two FMA chains per row
// (words 0-1 and 2-3), added at the end.
template <int OFF, int NS>
__device__ __forceinline__ void q4_block(const uint4 (&w)[NS], const float *xb, float2 (&blk)[NS])
{
    float2 a[NS], c[NS];
    {
        const float4 x0 = ld_xq4(xb, 0), x1 = ld_xq4(xb, 1);
#pragma unroll
        for (int i = 0; i < NS; ++i) a[i] = nib8_fma<OFF, true>(w[i].x, x0, x1, mk2(0.f, 0.f));
    }
    {
        const float4 x2 = ld_xq4(xb, 2), x3 = ld_xq4(xb, 3);
#pragma unroll
        for (int i = 0; i < NS; ++i) a[i] = nib8_fma<OFF, false>(w[i].y, x2, x3, a[i]);
    }
    {
        const float4 x4 = ld_xq4(xb, 4), x5 = ld_xq4(xb, 5);
#pragma unroll
        for (int i = 0; i < NS; ++i) c[i] = nib8_fma<OFF, true>(w[i].z, x4, x5, mk2(0.f, 0.f));
    }
    {
        const float4 x6 = ld_xq4(xb, 6), x7 = ld_xq4(xb, 7);
#pragma unroll
        for (int i = 0; i < NS; ++i) c[i] = nib8_fma<OFF, false>(w[i].w, x6, x7, c[i]);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) blk[i] = __fadd2_rn(a[i], c[i]);
}

// The same for offset-free codes against x staged by stage_x_q4k: the
// partial sums come out scaled by 2^-c.
template <int NS>
__device__ __forceinline__ void q4_block_sub(const uint4 (&w)[NS], const float *xb, float2 (&blk)[NS])
{
    float2 a[NS], c[NS];
    {
        const float4 x0 = ld_xq4(xb, 0), x1 = ld_xq4(xb, 1);
#pragma unroll
        for (int i = 0; i < NS; ++i) a[i] = nib8_sub_fma<true>(w[i].x, x0, x1, mk2(0.f, 0.f));
    }
    {
        const float4 x2 = ld_xq4(xb, 2), x3 = ld_xq4(xb, 3);
#pragma unroll
        for (int i = 0; i < NS; ++i) a[i] = nib8_sub_fma<false>(w[i].y, x2, x3, a[i]);
    }
    {
        const float4 x4 = ld_xq4(xb, 4), x5 = ld_xq4(xb, 5);
#pragma unroll
        for (int i = 0; i < NS; ++i) c[i] = nib8_sub_fma<true>(w[i].z, x4, x5, mk2(0.f, 0.f));
    }
    {
        const float4 x6 = ld_xq4(xb, 6), x7 = ld_xq4(xb, 7);
#pragma unroll
        for (int i = 0; i < NS; ++i) c[i] = nib8_sub_fma<false>(w[i].w, x6, x7, c[i]);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) blk[i] = __fadd2_rn(a[i], c[i]);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h)
{
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h)));
}

// ---------------------------------------------------------------- Q4_0
// Packed Q4_0: nibble plane (16 B per block, element order) + fp16 scale plane.
// One row task of NS rows: set the row pointers, prime() issues the loads of
// the first batch (U blocks of every row; a kernel may call it before
// waiting for the previous kernel, since weights never depend on it), run()
// computes each batch and then issues the next.  A batch is loaded whole
// before any of it is used, so a lane keeps U*NS 16-byte loads in flight and
// the SM as many bytes as its warps hold batches: HBM latency is covered by
// the bytes in flight (Little's law), not by a second register set.
template <int LG, int NS, int U>
struct Q40Stream {
    static constexpr int kStep = LG * U;
    const uint4 *wp[NS];     // row i's payload plus this lane's first block
    const uint16_t *sp[NS];  // row i's scales plus this lane's first block
    uint4 w[U][NS];
    uint32_t d[U][NS];

    // Batch [base, base + kStep) of the rows; kFull: wholly inside the row
    // (no bounds test).
    template <bool kFull>
    __device__ __forceinline__ void load(int base, int nb, int lp)
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kFull || base + lp + u * LG < nb) {
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    w[u][i] = ld_stream16(wp[i] + base + u * LG);
                    d[u][i] = ld_stream_u16(sp[i] + base + u * LG);
                }
            }
        }
    }
    template <bool kFull>
    __device__ __forceinline__ void compute(int base, int nb, int lp, const float *xs, float2 (&acc)[NS]) const
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = base + lp + u * LG;
            if (kFull || b < nb) {
                float2 blk[NS];
                q4_block<8, NS>(w[u], xs + b * kXBlk, blk);
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const float dd = half_bits_to_float(d[u][i]);
                    acc[i] = ffma2(blk[i], make_float2(dd, dd), acc[i]);
                }
            }
        }
    }
    __device__ __forceinline__ void prime(int nb, int lp)
    {
        if (kStep <= nb)
            load<true>(0, nb, lp);
        else
            load<false>(0, nb, lp);
    }
    __device__ __forceinline__ void run(const float *xs, int nb, int lp, float (&out)[NS])
    {
        float2 acc[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);
        for (int base = 0;;) {
            if (base + kStep <= nb)
                compute<true>(base, nb, lp, xs, acc);
            else
                compute<false>(base, nb, lp, xs, acc);
            base += kStep;
            if (base >= nb) break;
            if (base + kStep <= nb)
                load<true>(base, nb, lp);
            else
                load<false>(base, nb, lp);
        }
#pragma unroll
        for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
    }
};

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
// within the row), super-block sb/8, sub-block s = sb%8.  The staged x block
// carries the block's sum of x (for the min term).
//
// The 6-bit scale and min of sub-block s come from the record's scale bytes
// A = byte (s&3), B = byte (s&3)+4, C = byte (s&3)+8: sc = A&63, m = B&63
// for s < 4; sc = (C&15) | (A>>6)<<4, m = (C>>4) | (B>>6)<<4 for s >= 4.  A
// lane always sees the same s, so the shifts and masks are per-lane
// constants and the decode has no branch:
//   sc = ((y >> shA) & m1) | ((w >> shC) & m2)
//   m  = ((z >> shA) & m1) | ((w >> (shC+4)) & m2)
// with shA = 8(s&3) (+2 for s >= 4), shC = 8(s&3), m1 = 63 / 48, m2 = 0 / 15.
struct Q4KSub {
    int shA, shC;
    uint32_t m1, m2;
};
__device__ __forceinline__ Q4KSub q4k_sub(int s)
{
    Q4KSub c;
    c.shC = 8 * (s & 3);
    c.shA = c.shC + (s >= 4 ? 2 : 0);
    c.m1 = s >= 4 ? 48u : 63u;
    c.m2 = s >= 4 ? 15u : 0u;
    return c;
}
// d * sc and dmin * m of one sub-block (both exact in f32: 11-bit x 6-bit).
__device__ __forceinline__ void q4k_dm(uint4 rec, const Q4KSub &c, float &dsc, float &dm)
{
    const uint32_t isc = ((rec.y >> c.shA) & c.m1) | ((rec.w >> c.shC) & c.m2);
    const uint32_t imn = ((rec.z >> c.shA) & c.m1) | ((rec.w >> (c.shC + 4)) & c.m2);
    dsc = half_bits_to_float(rec.x & 0xFFFFu) * __uint2float_rn(isc);
    dm = half_bits_to_float(rec.x >> 16) * __uint2float_rn(imn);
}

// One row task of NS Q4_K rows, in the same batched prime() / run() form as
// Q40Stream, against x staged by stage_x_q4k (sums scaled by 2^-c).  The
// row pointers already point at this lane's first sub-block and super-block
// record; a batch covers sub-blocks [base, base + LG*U) of the rows, and
// batches that lie wholly inside the row skip every bounds test.
template <int LG, int NS, int U>
struct Q4KStream {
    static_assert(LG % 8 == 0, "a lane's sub-block position must be fixed");
    static constexpr int kStep = LG * U;
    const uint4 *wp[NS];
    const uint4 *rp[NS];
    uint4 w[U][NS], r[U][NS];

    template <bool kFull>
    __device__ __forceinline__ void load(int base, int nsb, int lp)
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kFull || base + lp + u * LG < nsb) {
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    w[u][i] = ld_stream16(wp[i] + base + u * LG);
                    // the 16-byte record is shared by the 8 lanes of a super-block
                    // (base is a multiple of 8: whole super-blocks)
                    r[u][i] = __ldg(rp[i] + (base >> 3) + u * (LG / 8));
                }
            }
        }
    }
    template <bool kFull>
    __device__ __forceinline__ void compute(int base, int nsb, int lp, const float *xs, const Q4KSub &sub,
                                            float2 (&acc)[NS]) const
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = base + lp + u * LG;
            if (kFull || b < nsb) {
                const float *xb = xs + b * kXBlk;
                float2 blk[NS];
                q4_block_sub<NS>(w[u], xb, blk);
                const float xsb = xb[32];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    float dsc, dm;
                    q4k_dm(r[u][i], sub, dsc, dm);
                    acc[i] = ffma2(blk[i], make_float2(dsc, dsc), acc[i]);
                    acc[i].x = fmaf(-dm, xsb, acc[i].x);
                }
            }
        }
    }
    __device__ __forceinline__ void prime(int nsb, int lp)
    {
        if (kStep <= nsb)
            load<true>(0, nsb, lp);
        else
            load<false>(0, nsb, lp);
    }
    __device__ __forceinline__ void run(const float *xs, int nsb, int lp, float (&out)[NS])
    {
        const Q4KSub sub = q4k_sub(lp & 7);
        float2 acc[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);
        for (int base = 0;;) {
            if (base + kStep <= nsb)
                compute<true>(base, nsb, lp, xs, sub, acc);
            else
                compute<false>(base, nsb, lp, xs, sub, acc);
            base += kStep;
            if (base >= nsb) break;
            if (base + kStep <= nsb)
                load<true>(base, nsb, lp);
            else
                load<false>(base, nsb, lp);
        }
#pragma unroll
        for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
    }
};

// ---------------------------------------------------------------- kernel-side common
constexpr int kThreadsPerCta = 256;
constexpr int kWarpsPerCta = kThreadsPerCta / 32;

// The row tasks (TR rows each) of one warp: rows start + j*step .. for
// j < count, then (balanced schedule only) ntail rows from tail_begin that
// all warps of the CTA share along K.
//   round-robin: task t of the grid goes to warp t % (warps in the grid); the
//     last round may be partly filled (rows past the end are not stored).
//   balanced: each CTA takes a near-equal contiguous share of the rows; its
//     warps process whole tasks while every warp has one, and the fewer than
//     kWarpsPerCta*TR rows left are split along K (warp w takes the w-th
//     eighth of the blocks), their partial sums added in shared memory in
//     warp order.  Chosen by the host when round-robin would leave a sparse
//     last round with most warps idle (fewer than ~1.75 tasks per warp).
struct WarpRows {
    int start, step, count, tail_begin, ntail;
};
template <int TR>
__device__ __forceinline__ WarpRows warp_rows(int rows, bool balanced, int warp)
{
    WarpRows c;
    if (balanced) {
        const int lo = rows / static_cast<int>(gridDim.x), extra = rows % static_cast<int>(gridDim.x);
        const int b = static_cast<int>(blockIdx.x);
        const int begin = b * lo + min(b, extra);
        const int n = lo + (b < extra ? 1 : 0);
        c.count = n / (kWarpsPerCta * TR);
        c.start = begin + warp * TR;
        c.step = kWarpsPerCta * TR;
        c.tail_begin = begin + c.count * kWarpsPerCta * TR;
        c.ntail = n - c.count * kWarpsPerCta * TR;
    } else {
        const int ntasks = (rows + TR - 1) / TR;
        const int first = static_cast<int>(blockIdx.x) * kWarpsPerCta + warp;
        const int stride = static_cast<int>(gridDim.x) * kWarpsPerCta;
        c.count = first < ntasks ? (ntasks - 1 - first) / stride + 1 : 0;
        c.start = first * TR;
        c.step = stride * TR;
        c.tail_begin = 0;
        c.ntail = 0;
    }
    return c;
}
// Blocks [lo, hi) of warp w for the tail rows; slice edges are multiples of
// `align` blocks (nb % align == 0).
__device__ __forceinline__ void tail_slice(int nb, int align, int w, int &lo, int &hi)
{
    const int units = nb / align;
    lo = (units * w / kWarpsPerCta) * align;
    hi = (units * (w + 1) / kWarpsPerCta) * align;
}

// Ask L2 for the weights of the TR-row task starting at row r0: lane i < TR
// prefetches row r0 + i of the payload plane (row_bytes each, a multiple of
// 16); lane 31 prefetches the rows' scale records, one contiguous range of
// the scale plane (row_sc bytes per row) rounded to 16-byte boundaries that
// stay inside the plane.  A prefetch is only a hint: the loads that follow
// read the same bytes whether or not it has landed.
template <int TR>
__device__ __forceinline__ void prefetch_task_l2(const uint8_t *pay, uint32_t row_bytes, const uint8_t *sc,
                                                 uint32_t row_sc, int r0, int rows, int lane)
{
    if (lane < TR && r0 + lane < rows) prefetch_l2_bulk(pay + static_cast<size_t>(r0 + lane) * row_bytes, row_bytes);
    if (lane == 31 && r0 < rows) {
        const size_t plane = static_cast<size_t>(rows) * row_sc;
        const size_t lo = (static_cast<size_t>(r0) * row_sc) & ~static_cast<size_t>(15);
        size_t hi = static_cast<size_t>(min(r0 + TR, rows)) * row_sc;
        hi = (hi + 15) & ~static_cast<size_t>(15);
        const size_t cap = plane & ~static_cast<size_t>(15);
        if (hi > cap) hi = cap;
        if (hi > lo) prefetch_l2_bulk(sc + lo, static_cast<uint32_t>(hi - lo));
    }
}

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
// the 4-bit streams also take eight-block batches
#define GQ_GEO_CASE1B(geo, CASE, LG, R)                                 \
    GQ_GEO_CASE1(geo, CASE, LG, R)                                      \
    if ((geo).lg == LG && (geo).r == R && (geo).u == 8) { CASE(LG, R, 8); }
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
#ifdef GQ_TUNING
#define GQ_GEO_TUNING_CASES(geo, CASE)                                              \
    if ((geo).lg == 8 && (geo).r == 4 && (geo).u == 4) { CASE(8, 4, 4); }          \
    if ((geo).lg == 16 && (geo).r == 4 && (geo).u == 4) { CASE(16, 4, 4); }        \
    if ((geo).lg == 32 && (geo).r == 4 && (geo).u == 4) { CASE(32, 4, 4); }        \
    if ((geo).lg == 8 && (geo).r == 4 && (geo).u == 2) { CASE(8, 4, 2); }
#else
#define GQ_GEO_TUNING_CASES(geo, CASE)
#endif
#define GQ_GEO_SWITCH_R12(geo, CASE)          \
    do {                                      \
        GQ_GEO_CASE1B(geo, CASE, 32, 1)        \
        GQ_GEO_CASE1B(geo, CASE, 32, 2)        \
        GQ_GEO_CASE1B(geo, CASE, 16, 1)        \
        GQ_GEO_CASE1B(geo, CASE, 16, 2)        \
        GQ_GEO_CASE1B(geo, CASE, 8, 1)         \
        GQ_GEO_CASE1B(geo, CASE, 8, 2)         \
        GQ_GEO_TUNING_CASES(geo, CASE)        \
        return GQ_ERR_SHAPE;                  \
    } while (0)
