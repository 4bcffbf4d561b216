// gq_q6k.cu -- Q6_K x f32 decode matvec.
//
// "Metal kernel capability table (Phase B ground truth)", section 1:
// q6k_matvec (210-byte super-blocks, K % 256, rows masked; here K % 256 is
// checked at dispatch).  Within a super-block of 256 weights,
//   w_j = d * sc[j / 16] * (q_j - 32),  q_j = lo_j + 16 * hi_j  (6 bits)
// with the packed planes: low 4 bits in element order (16 bytes per 32
// weights), top 2 bits four to a byte (8 bytes per 32 weights), and 18-byte
// records {16 int8 sub-scales, fp16 d}.
//
// Layout of the work: lane groups of LG lanes take R rows; lane p takes the
// 32-weight chunks p, p + LG, ... of the row (LG is a multiple of 8, so a
// lane's chunk always holds the same two sub-blocks of its super-blocks).
// Per chunk a lane loads 16 bytes of low bits and 8 bytes of top bits; the
// x vector is staged once per CTA in the 4-bit kernels' permuted blocks.
//
// Exact codes without per-element shifts: for the element pair (e, e + 4) of
// an 8-element group, OR-ing the masked low nibble into the f32 pattern of
// 2^23 gives A = 2^23 + lo * 16^e and the masked top bits B = 2^23 + hi * 4^e
// (both exact); then
//   R = B * 16 * 4^-e - (2^23 * 16^-e + 2^27 * 4^-e + 32) = 16 hi - 2^23 16^-e - 32
//   v = A * 16^-e + R = lo + 16 hi - 32
// are each one FMA whose exact result is representable, so v is exact.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {
namespace q6 {

// Sum over one 8-element group of v_j * x_j as a pair of partial sums (the
// pair order of the staged x): w = the group's 8 low nibbles (element m at
// bits 4m), h = its 8 top-bit pairs (element m at bits 2m), x8 = the staged
// x of the group.
__device__ __forceinline__ float2 group_dot(uint32_t w, uint32_t h, const float *x8, float2 acc)
{
    const uint32_t w2 = w >> 16, h2 = h >> 8;
    const float4 xa = ld_xq4(x8, 0), xb = ld_xq4(x8, 1);
    const float2 xp[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w), make_float2(xb.x, xb.y),
                          make_float2(xb.z, xb.w)};
    // per e: 16^-e, 16 * 4^-e, -(2^23 16^-e + 2^27 4^-e + 32)
    const float sl[4] = {1.0f, 0.0625f, 0.00390625f, 0.000244140625f};
    const float sh[4] = {16.0f, 4.0f, 1.0f, 0.25f};
    const float cc[4] = {-(8388608.0f + 134217728.0f + 32.0f), -(524288.0f + 33554432.0f + 32.0f),
                         -(32768.0f + 8388608.0f + 32.0f), -(2048.0f + 2097152.0f + 32.0f)};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t ml = 0xFu << (4 * e), mh = 3u << (2 * e);
        const float2 A = make_float2(__uint_as_float((w & ml) | 0x4B000000u), __uint_as_float((w2 & ml) | 0x4B000000u));
        const float2 B = make_float2(__uint_as_float((h & mh) | 0x4B000000u), __uint_as_float((h2 & mh) | 0x4B000000u));
        const float2 R = __ffma2_rn(B, make_float2(sh[e], sh[e]), make_float2(cc[e], cc[e]));
        const float2 v = __ffma2_rn(A, make_float2(sl[e], sl[e]), R);
        acc = __ffma2_rn(v, xp[e], acc);
    }
    return acc;
}

template <int LG, int R, int U>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q6k_matvec(const uint4 *__restrict__ lo, const uint2 *__restrict__ hi, const uint8_t *__restrict__ rec,
                 const float *__restrict__ x, float *__restrict__ y, int rows, int nsb)
{
    static_assert(LG % 8 == 0, "a lane's sub-blocks must be fixed");
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ns = nsb >> 3;
    const int sub = 2 * (lp & 7);  // the first of this lane's two sub-blocks in a super-block
    const int ntasks = (rows + TR - 1) / TR;
    const int first = blockIdx.x * kWarpsPerCta + warp;
    const int stride = gridDim.x * kWarpsPerCta;

    if (first < ntasks) {  // weights never depend on the previous kernel
        const void *rp[TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) rp[i] = lo + static_cast<size_t>(min(first * TR + i, rows - 1)) * nsb;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
    }
    pdl_wait();
    stage_x_q4<false>(xs, x, nsb * 32);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += stride) {
        int r[R];
#pragma unroll
        for (int i = 0; i < R; ++i) r[i] = min(task * TR + g * R + i, rows - 1);
        float2 acc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = make_float2(0.f, 0.f);
        for (int b0 = lp; b0 < nsb; b0 += LG * U) {
            uint4 wl[U][R];
            uint2 wh[U][R];
            float dsc[U][R][2];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int b = b0 + u * LG;
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    if (b < nsb) {
                        const size_t c = static_cast<size_t>(r[i]) * nsb + b;
                        wl[u][i] = ld_stream16(lo + c);
                        wh[u][i] = __ldg(hi + c);
                        const uint8_t *rc = rec + (static_cast<size_t>(r[i]) * ns + (b >> 3)) * 18;
                        const uint32_t scp = __ldg(reinterpret_cast<const uint16_t *>(rc + sub));
                        const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const uint16_t *>(rc + 16))));
                        dsc[u][i][0] = d * static_cast<float>(static_cast<int8_t>(scp & 0xFFu));
                        dsc[u][i][1] = d * static_cast<float>(static_cast<int8_t>(scp >> 8));
                    } else {
                        wl[u][i] = make_uint4(0u, 0u, 0u, 0u);
                        wh[u][i] = make_uint2(0u, 0u);
                        dsc[u][i][0] = dsc[u][i][1] = 0.f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int b = b0 + u * LG;
                if (b < nsb) {
                    const float *xb = xs + b * kXBlk;
#pragma unroll
                    for (int i = 0; i < R; ++i) {
                        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
                        s0 = group_dot(wl[u][i].x, wh[u][i].x & 0xFFFFu, xb, s0);
                        s0 = group_dot(wl[u][i].y, wh[u][i].x >> 16, xb + 8, s0);
                        s1 = group_dot(wl[u][i].z, wh[u][i].y & 0xFFFFu, xb + 16, s1);
                        s1 = group_dot(wl[u][i].w, wh[u][i].y >> 16, xb + 24, s1);
                        acc[i] = __ffma2_rn(s0, make_float2(dsc[u][i][0], dsc[u][i][0]), acc[i]);
                        acc[i] = __ffma2_rn(s1, make_float2(dsc[u][i][1], dsc[u][i][1]), acc[i]);
                    }
                }
            }
        }
        const int r0 = task * TR + g * R;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(acc[i].x + acc[i].y);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

}  // namespace q6

int launch_q6k_matvec(const void *W, const float *x, float *y, int rows, int K, cudaStream_t s)
{
    constexpr int LG = 16, R = 2, U = 2;
    const int nsb = K / 32, ns = K / 256;
    const uint8_t *base = static_cast<const uint8_t *>(W);
    const uint4 *lo = reinterpret_cast<const uint4 *>(base);
    const uint2 *hi = reinterpret_cast<const uint2 *>(base + static_cast<size_t>(rows) * ns * 128);
    const uint8_t *rec = base + static_cast<size_t>(rows) * ns * 192;
    const size_t smem = static_cast<size_t>(nsb) * kXBlk * sizeof(float);
    const long long ntasks = (rows + (32 / LG) * R - 1) / ((32 / LG) * R);
    auto kern = q6::k_q6k_matvec<LG, R, U>;
    const int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks);
    if (grid <= 0) return GQ_ERR_SHAPE;
    return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, lo, hi, rec, x, y, rows, nsb));
}

}  // namespace gq
