// gq_q4_0.cu -- Q4_0 x f32 decode matvec.
//
// "Gemma 4 M4 Max kernel roadmap", K2 "Metal decode path", step 1: direct
// Q4_0 matrix-vector product with fused dequantization and F32
// accumulation.  "Metal kernel capability table (Phase B ground truth)",
// section 1, q4_f32_matvec (rows masked; here K is never truncated).
//
// Persistent kernel: each CTA stages x once (swizzled, cp.async), then its
// warps stream packed Q4_0 rows (16-byte nibble loads + fp16 scales); see
// gq_matvec.cuh for the lane geometry and the exact nibble-to-f32 step.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U, int P>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4_0_matvec(const uint4 *__restrict__ nib, const uint16_t *__restrict__ dsc,
                  const float *__restrict__ x, float *__restrict__ y, int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const int first = blockIdx.x * kWarpsPerCta + warp;

    if (first < ntasks) {
        const void *rp[TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(first * TR + i, rows - 1)) * nb;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
    }
    pdl_wait();
    stage_x_perm8(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += gridDim.x * kWarpsPerCta) {
        const int r0 = task * TR + g * R;
        const uint4 *wp[R];
        const uint16_t *sp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(r0 + i, rows - 1);
            wp[i] = nib + static_cast<size_t>(r) * nb;
            sp[i] = dsc + static_cast<size_t>(r) * nb;
        }
        float out[R];
        if (P == 2)
            q4_0_stream2<LG, R, U>(wp, sp, xs, nb, lp, out);
        else
            q4_0_stream<LG, R, U>(wp, sp, xs, nb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(out[i]);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

int launch_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                 \
    {                                                                                                  \
        auto kern = k_q4_0_matvec<LG, R, U, PP>;                                                       \
        const int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                            \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, nib, dsc, x, y, rows, nb)); \
    }
    if (geo.p == 2) {
        constexpr int PP = 2;
        GQ_PAIR_SWITCH(geo, CASE);
    } else {
        constexpr int PP = 1;
        GQ_GEO_SWITCH(geo, CASE);
    }
#undef CASE
}

}  // namespace gq
