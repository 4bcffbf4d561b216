// gq_q4k.cu -- Q4_K x f32 decode matvec.
//
// "Metal kernel capability table (Phase B ground truth)", section 1:
// q4k_matvec / q4k_matvec_8sg (144-byte super-blocks, K % 256, rows masked;
// here K % 256 is asserted at dispatch rather than assumed).
//   y_i = sum over super-blocks and sub-blocks s of
//         d*sc_s * sum_j q_j x_j  -  dmin*m_s * sum_j x_j
// The per-32 sums of x are computed once per CTA next to the staged x.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U, int P>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4k_matvec(const uint4 *__restrict__ nib, const uint4 *__restrict__ rec,
                 const float *__restrict__ x, float *__restrict__ y, int rows, int nsb)
{
    extern __shared__ __align__(16) float xs[];
    float *xsum = xs + nsb * 32;
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const int ns = nsb >> 3;
    const int first = blockIdx.x * kWarpsPerCta + warp;

    if (first < ntasks) {
        const void *rp[TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(first * TR + i, rows - 1)) * nsb;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
    }
    pdl_wait();
    stage_x_perm8(xs, x, nsb * 32);
    stage_xsum(xsum, xs, nsb);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += gridDim.x * kWarpsPerCta) {
        const int r0 = task * TR + g * R;
        const uint4 *wp[R];
        const uint4 *rp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(r0 + i, rows - 1);
            wp[i] = nib + static_cast<size_t>(r) * nsb;
            rp[i] = rec + static_cast<size_t>(r) * ns;
        }
        float out[R];
        if (P == 2)
            q4k_stream2<LG, R, U>(wp, rp, xs, xsum, nsb, lp, out);
        else
            q4k_stream<LG, R, U>(wp, rp, xs, xsum, nsb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(out[i]);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

int launch_q4k_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                      cudaStream_t s)
{
    const int nsb = K / 32;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint4 *rec = nib + static_cast<size_t>(rows) * nsb;
    const size_t smem = static_cast<size_t>(K) * sizeof(float) + static_cast<size_t>(nsb) * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                 \
    {                                                                                                  \
        auto kern = k_q4k_matvec<LG, R, U, PP>;                                                        \
        const int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                            \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, nib, rec, x, y, rows, nsb)); \
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
