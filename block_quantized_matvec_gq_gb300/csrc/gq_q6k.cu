// gq_q6k.cu -- Q6_K x f32 decode matvec.
//
// "Metal kernel capability table (Phase B ground truth)", section 1:
// q6k_matvec (210-byte super-blocks, K % 256, rows masked; here K % 256 is
// checked at dispatch).  Within a super-block of 256 weights,
//   w_j = d * sc[j / 16] * (q_j - 32),  q_j = lo_j + 16 * hi_j  (6 bits)
// with the packed planes (gq_pack): low 4 bits in element order (16 bytes per
// 32 weights), top 2 bits as one 32-bit word per 16 weights arranged for the
// decode below, 16-byte int8 sub-scale records, fp16 d.
//
// Exact codes, two LOP3s per element and one bit-select per two: for the
// four elements of a 16-bit half of a low-bit word (nibble i at bits 4i), the
// top-bit word shifted by the half's amount (+4, +2, -12 or -14, per the
// packed arrangement) holds each element's two top bits at bits 4i + 4.  A
// bit-select taking bits {4,5, 12,13} from the shifted top bits and the rest
// from the low bits leaves elements 0 and 2 as 6-bit fields at bits 0..5 and
// 8..13; one taking bits {8,9, 16,17} leaves elements 1 and 3 at 4..9 and
// 12..17.  Each field then goes into the significand of 2^(23-4i) by one
// mask-and-OR (bit 4i on the units place, as for the 4-bit codes), giving
// 2^(23-4i) + q exactly; one packed add of -(2^(23-4i) + 32) leaves q - 32
// for the element pair (i, i+4), and one packed FMA adds its products.
//
// Layout of the work as in the 4-bit streams: lane groups of LG lanes take R
// rows; lane p takes the 32-weight chunks p, p + LG, ... of the row (LG a
// multiple of 8, so a lane's chunk is always the same eighth of its
// super-blocks); the x vector is staged once per CTA in the 4-bit kernels'
// permuted blocks.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {
namespace q6 {

#define GQ_Q6_GROUP_BODY(FIRST)                                                                                 \
    "{\n"                                                                                                       \
    " .reg .b32 wh, e0, o0, e1, o1, l0, h0, l1, h1, l2, h2, l3, h3;\n"                                         \
    " .reg .b64 p0, p1, p2, p3, x0, x1, x2, x3, a, c0, c1, c2, c3;\n"                                          \
    " shr.u32 wh, %2, 16;\n"                                                                                    \
    " lop3.b32 e0, %2, %3, 0x00003030, 0xD8;\n lop3.b32 o0, %2, %3, 0x00030300, 0xD8;\n"                        \
    " lop3.b32 e1, wh, %4, 0x00003030, 0xD8;\n lop3.b32 o1, wh, %4, 0x00030300, 0xD8;\n"                        \
    " lop3.b32 l0, e0, 0x0000003F, 0x4B000000, 0xEA;\n lop3.b32 h0, e1, 0x0000003F, 0x4B000000, 0xEA;\n"        \
    " lop3.b32 l1, o0, 0x000003F0, 0x49000000, 0xEA;\n lop3.b32 h1, o1, 0x000003F0, 0x49000000, 0xEA;\n"        \
    " lop3.b32 l2, e0, 0x00003F00, 0x47000000, 0xEA;\n lop3.b32 h2, e1, 0x00003F00, 0x47000000, 0xEA;\n"        \
    " lop3.b32 l3, o0, 0x0003F000, 0x45000000, 0xEA;\n lop3.b32 h3, o1, 0x0003F000, 0x45000000, 0xEA;\n"        \
    " mov.b64 p0, {l0, h0};\n mov.b64 p1, {l1, h1};\n mov.b64 p2, {l2, h2};\n mov.b64 p3, {l3, h3};\n"        \
    " mov.b64 c0, {%15, %15};\n mov.b64 c1, {%16, %16};\n mov.b64 c2, {%17, %17};\n mov.b64 c3, {%18, %18};\n" \
    " add.rn.f32x2 p0, p0, c0;\n add.rn.f32x2 p1, p1, c1;\n add.rn.f32x2 p2, p2, c2;\n add.rn.f32x2 p3, p3, c3;\n" \
    " mov.b64 x0, {%5, %6};\n mov.b64 x1, {%7, %8};\n mov.b64 x2, {%9, %10};\n mov.b64 x3, {%11, %12};\n"      \
    " mov.b64 a, {%13, %14};\n" FIRST                                                                           \
    " fma.rn.f32x2 a, p1, x1, a;\n fma.rn.f32x2 a, p2, x2, a;\n fma.rn.f32x2 a, p3, x3, a;\n"                  \
    " mov.b64 {%0, %1}, a;\n"                                                                                   \
    "}"

// acc + sum over one 8-element group of (q - 32) * x as a packed pair of
// partial sums: w = the group's low-bit word, hl / hh = its top-bit word
// shifted for the low / high half; xa, xb = the staged x of the group.
template <bool kStart>
__device__ __forceinline__ float2 group_fma(uint32_t w, uint32_t hl, uint32_t hh, float4 xa, float4 xb, float2 acc)
{
    float2 r;
    if (kStart) {
        asm(GQ_Q6_GROUP_BODY(" mul.rn.f32x2 a, p0, x0;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "r"(hl), "r"(hh), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y),
              "f"(xb.z), "f"(xb.w), "f"(acc.x), "f"(acc.y), "f"(NibConsts<32>::c0), "f"(NibConsts<32>::c1),
              "f"(NibConsts<32>::c2), "f"(NibConsts<32>::c3));
    } else {
        asm(GQ_Q6_GROUP_BODY(" fma.rn.f32x2 a, p0, x0, a;\n")
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "r"(hl), "r"(hh), "f"(xa.x), "f"(xa.y), "f"(xa.z), "f"(xa.w), "f"(xb.x), "f"(xb.y),
              "f"(xb.z), "f"(xb.w), "f"(acc.x), "f"(acc.y), "f"(NibConsts<32>::c0), "f"(NibConsts<32>::c1),
              "f"(NibConsts<32>::c2), "f"(NibConsts<32>::c3));
    }
    return r;
}

// One 16-weight sub-block: low-bit words w0 (elements 0-7), w1 (8-15), their
// top-bit word h; x16 = the staged x of the 16 elements.
__device__ __forceinline__ float2 sub_dot(uint32_t w0, uint32_t w1, uint32_t h, const float *x16)
{
    float2 s = group_fma<true>(w0, h << 4, h << 2, ld_xq4(x16, 0), ld_xq4(x16, 1), make_float2(0.f, 0.f));
    return group_fma<false>(w1, h >> 12, h >> 14, ld_xq4(x16, 2), ld_xq4(x16, 3), s);
}

// d * sc for the chunk's two sub-blocks: s16 = their int8 scales (low byte
// first), dh = fp16 d.  The bytes become exact floats through 2^23 + (sc + 128).
__device__ __forceinline__ float2 chunk_scales(uint32_t s16, uint32_t dh)
{
    const uint32_t u = s16 ^ 0x8080u;
    const float2 sc = __fadd2_rn(mk2(byte_f(u, 0x7540u), byte_f(u, 0x7541u)),
                                 mk2(-(0x1p23f + 128.0f), -(0x1p23f + 128.0f)));
    const float d = half_bits_to_float(dh);
    return __fmul2_rn(sc, mk2(d, d));
}

struct Planes {
    const uint4 *lo;      // rows * nsb chunks of low bits
    const uint2 *hi;      // rows * nsb chunks of top bits
    const uint16_t *sc;   // rows * nsb pairs of sub-scales
    const uint16_t *d;    // rows * ns fp16 d
};

// One row task of NS rows: ci[i] = the index of this lane's first chunk of
// row i in the three chunk planes (low bits, top bits, pair of sub-scales),
// di[i] = that of its super-block in the d plane; a batch covers chunks
// [base, base + LG*U) of the rows, and batches wholly inside the row skip
// every bounds test.
template <int LG, int NS, int U>
struct Q6KStream {
    static_assert(LG % 8 == 0, "a lane's chunk position in the super-block must be fixed");
    static constexpr int kStep = LG * U;
    uint32_t ci[NS], di[NS];
    uint4 w[U][NS];
    uint2 h[U][NS];
    uint32_t s[U][NS], d[U][NS];

    template <bool kFull>
    __device__ __forceinline__ void load(const Planes &pl, int base, int nsb, int lp)
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (kFull || base + lp + u * LG < nsb) {
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const uint32_t c = ci[i] + static_cast<uint32_t>(base + u * LG);
                    w[u][i] = ld_stream16(pl.lo + c);
                    h[u][i] = __ldg(pl.hi + c);
                    s[u][i] = __ldg(pl.sc + c);
                    // base is a multiple of 8 (whole super-blocks)
                    d[u][i] = __ldg(pl.d + di[i] + static_cast<uint32_t>((base >> 3) + u * (LG / 8)));
                }
            }
        }
    }
    template <bool kFull>
    __device__ __forceinline__ void compute(int base, int nsb, int lp, const float *xs, float2 (&acc)[NS]) const
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = base + lp + u * LG;
            if (kFull || b < nsb) {
                const float *xb = xs + b * kXBlk;
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    const float2 s0 = sub_dot(w[u][i].x, w[u][i].y, h[u][i].x, xb);
                    const float2 s1 = sub_dot(w[u][i].z, w[u][i].w, h[u][i].y, xb + 16);
                    const float2 ds = chunk_scales(s[u][i], d[u][i]);
                    acc[i] = ffma2(s0, mk2(ds.x, ds.x), acc[i]);
                    acc[i] = ffma2(s1, mk2(ds.y, ds.y), acc[i]);
                }
            }
        }
    }
    __device__ __forceinline__ void prime(const Planes &pl, int nsb, int lp)
    {
        if (kStep <= nsb)
            load<true>(pl, 0, nsb, lp);
        else
            load<false>(pl, 0, nsb, lp);
    }
    __device__ __forceinline__ void run(const Planes &pl, const float *xs, int nsb, int lp, float (&out)[NS])
    {
        float2 acc[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) acc[i] = make_float2(0.f, 0.f);
        for (int base = 0;;) {
            if (base + kStep <= nsb)
                compute<true>(base, nsb, lp, xs, acc);
            else
                compute<false>(base, nsb, lp, xs, acc);
            base += kStep;
            if (base >= nsb) break;
            if (base + kStep <= nsb)
                load<true>(pl, base, nsb, lp);
            else
                load<false>(pl, base, nsb, lp);
        }
#pragma unroll
        for (int i = 0; i < NS; ++i) out[i] = acc[i].x + acc[i].y;
    }
};

// Rows r0 + g*R + i (clamped to the last row) of a task, chunks from blo
// (a multiple of 8).
template <int LG, int R, int U>
__device__ __forceinline__ void setup_rows(Q6KStream<LG, R, U> &st, int r0, int g, int lp, int rows, int nsb, int blo)
{
    const int ns = nsb >> 3;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const uint32_t r = static_cast<uint32_t>(min(r0 + g * R + i, rows - 1));
        st.ci[i] = r * static_cast<uint32_t>(nsb) + static_cast<uint32_t>(blo + lp);
        st.di[i] = r * static_cast<uint32_t>(ns) + static_cast<uint32_t>((blo + lp) >> 3);
    }
}

// The next task's rows into L2: low and top bits (lanes < TR, lane 31), then
// sub-scales and d.
template <int TR>
__device__ __forceinline__ void prefetch_task(const Planes &pl, int nsb, int r0, int rows, int lane)
{
    prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(pl.lo), nsb * 16u, reinterpret_cast<const uint8_t *>(pl.hi),
                         nsb * 8u, r0, rows, lane);
    prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(pl.sc), nsb * 2u, reinterpret_cast<const uint8_t *>(pl.d),
                         (nsb >> 3) * 2u, r0, rows, lane);
}

template <int LG, int R, int U, int kMode>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q6k_matvec(Planes pl, const float *__restrict__ x, float *__restrict__ y, int rows, int nsb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    // schedule (chosen by the host): 0 round-robin; 1 balanced; 2 balanced, first loads early
    constexpr bool kBalanced = kMode >= 1, kEarly = kMode == 2;
    __shared__ float part[kWarpsPerCta][kWarpsPerCta * TR];  // tail partial sums [warp][row]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    Q6KStream<LG, R, U> st;
    if constexpr (!kBalanced) {
        const int ntasks = (rows + TR - 1) / TR;
        const int first = blockIdx.x * kWarpsPerCta + warp;
        const int stride = gridDim.x * kWarpsPerCta;
        // weights never depend on the previous kernel: this warp's first rows
        // stream into L2 before waiting for it
        if (first < ntasks) {
            const void *rp[TR];
#pragma unroll
            for (int i = 0; i < TR; ++i) rp[i] = pl.lo + static_cast<size_t>(min(first * TR + i, rows - 1)) * nsb;
            prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
        }
        pdl_wait();
        stage_x_q4<false>(xs, x, nsb * 32);
        pdl_launch_dependents();
        for (int task = first; task < ntasks; task += stride) {
            setup_rows(st, task * TR, g, lp, rows, nsb, 0);
            st.prime(pl, nsb, lp);
            if (task + stride < ntasks) prefetch_task<TR>(pl, nsb, (task + stride) * TR, rows, lane);
            float out[R];
            st.run(pl, xs, nsb, lp, out);
            const int r0 = task * TR + g * R;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
            }
        }
    } else {
        const WarpRows cr = warp_rows<TR>(rows, kBalanced, warp);
        if (cr.count > 0) {
            const void *rp[TR];
#pragma unroll
            for (int i = 0; i < TR; ++i) rp[i] = pl.lo + static_cast<size_t>(min(cr.start + i, rows - 1)) * nsb;
            prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
            if (kEarly) {
                setup_rows(st, cr.start, g, lp, rows, nsb, 0);
                st.prime(pl, nsb, lp);
            }
        }
        pdl_wait();
        stage_x_q4<false>(xs, x, nsb * 32);
        pdl_launch_dependents();
        for (int j = 0; j < cr.count; ++j) {
            const int r0 = cr.start + j * cr.step;
            if (j > 0 || !kEarly) {
                setup_rows(st, r0, g, lp, rows, nsb, 0);
                st.prime(pl, nsb, lp);
            }
            if (j + 1 < cr.count) prefetch_task<TR>(pl, nsb, r0 + cr.step, rows, lane);
            float out[R];
            st.run(pl, xs, nsb, lp, out);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + g * R + i < rows) y[r0 + g * R + i] = s;
            }
        }
        if (cr.ntail > 0) {
            int blo, bhi;
            tail_slice(nsb, 8, warp, blo, bhi);
            for (int t0 = 0; t0 < cr.ntail; t0 += TR) {
                setup_rows(st, cr.tail_begin + t0, g, lp, rows, nsb, blo);
                st.prime(pl, bhi - blo, lp);
                float out[R];
                st.run(pl, xs + blo * kXBlk, bhi - blo, lp, out);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float s = group_sum<LG>(out[i]);
                    if (lp == 0) part[warp][t0 + g * R + i] = s;
                }
            }
            __syncthreads();
            for (int r = threadIdx.x; r < cr.ntail; r += kThreadsPerCta) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kWarpsPerCta; ++w) s += part[w][r];
                y[cr.tail_begin + r] = s;
            }
        }
    }
}

}  // namespace q6

int launch_q6k_matvec(const void *W, const float *x, float *y, int rows, int K, cudaStream_t s)
{
    const int nsb = K / 32, ns = K / 256;
    const uint8_t *base = static_cast<const uint8_t *>(W);
    const size_t sup = static_cast<size_t>(rows) * ns;
    q6::Planes pl;
    pl.lo = reinterpret_cast<const uint4 *>(base);
    pl.hi = reinterpret_cast<const uint2 *>(base + sup * 128);
    pl.sc = reinterpret_cast<const uint16_t *>(base + sup * 192);
    pl.d = reinterpret_cast<const uint16_t *>(base + sup * 208);
    const size_t smem = static_cast<size_t>(nsb) * kXBlk * sizeof(float);
    const MatvecGeo geo = choose_q6k_geo();
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                        \
    {                                                                                                         \
        auto rr = q6::k_q6k_matvec<LG, R, U, 0>;                                                              \
        int grid = persistent_grid(reinterpret_cast<const void *>(rr), kThreadsPerCta, smem, ntasks);        \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                                   \
        const long long w5 = static_cast<long long>(grid) * kWarpsPerCta;                                     \
        const int mode = schedule_mode(ntasks, w5, nsb);                                                           \
        auto kern = mode == 2 ? q6::k_q6k_matvec<LG, R, U, 2> : (mode == 1 ? q6::k_q6k_matvec<LG, R, U, 1> : rr); \
        if (mode != 0) { /* size through the launched instantiation too (raises its shared-memory limit) */  \
            const int g2 = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
            if (g2 <= 0) return GQ_ERR_SHAPE;                                                                 \
            if (g2 < grid) grid = g2;                                                                         \
        }                                                                                                     \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, pl, x, y, rows, nsb)); \
    }
    if (geo.lg == 16 && geo.r == 2 && geo.u == 4) CASE(16, 2, 4);
#ifdef GQ_TUNING
    if (geo.lg == 16 && geo.r == 2 && geo.u == 2) CASE(16, 2, 2);
    if (geo.lg == 16 && geo.r == 1 && geo.u == 4) CASE(16, 1, 4);
    if (geo.lg == 8 && geo.r == 2 && geo.u == 4) CASE(8, 2, 4);
    if (geo.lg == 32 && geo.r == 2 && geo.u == 2) CASE(32, 2, 2);
    if (geo.lg == 32 && geo.r == 1 && geo.u == 4) CASE(32, 1, 4);
#endif
#undef CASE
    return GQ_ERR_SHAPE;
}

}  // namespace gq
