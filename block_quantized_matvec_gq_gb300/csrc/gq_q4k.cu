// gq_q4k.cu -- Q4_K x f32 decode matvec.
//
// "Metal kernel capability table (Phase B ground truth)", section 1:
// q4k_matvec / q4k_matvec_8sg (144-byte super-blocks, K % 256, rows masked;
// here K % 256 is asserted at dispatch rather than assumed).
//   y_i = sum over super-blocks and sub-blocks s of
//         d*sc_s * sum_j q_j x_j  -  dmin*m_s * sum_j x_j
// The per-32 sums of x are computed once per CTA, inside the staged x blocks.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U, bool kEarly>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4k_matvec(const uint4 *__restrict__ nib, const uint4 *__restrict__ rec,
                 const float *__restrict__ x, float *__restrict__ y, int rows, int nsb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const int ns = nsb >> 3;
    const int first = blockIdx.x * kWarpsPerCta + warp;
    const int stride = gridDim.x * kWarpsPerCta;

    Q4KStream<LG, R, U> st;
    auto setup = [&](int task) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(task * TR + g * R + i, rows - 1);
            st.wp[i] = nib + static_cast<size_t>(r) * nsb;
            st.rp[i] = rec + static_cast<size_t>(r) * ns;
        }
        st.prime(nsb, lp);
    };
    // Weights never depend on the previous kernel: prefetch this warp's first
    // rows into L2 before waiting for it and, when warps have about one task
    // each (kEarly, chosen by the host), issue that task's first loads too.
    // (Measured: with several tasks per warp the early loads cost more than
    // they save.)
    if (first < ntasks) {
        const void *rp[TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(first * TR + i, rows - 1)) * nsb;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
        if (kEarly) setup(first);
    }
    pdl_wait();
    stage_x_q4<true>(xs, x, nsb * 32);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += stride) {
        if (task != first || !kEarly) setup(task);
        float out[R];
        st.run(xs, nsb, lp, out);
        const int r0 = task * TR + g * R;
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
    const size_t smem = static_cast<size_t>(nsb) * kXBlk * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
    if (geo.p != 1) return GQ_ERR_SHAPE;
#define CASE(LG, R, U)                                                                                  \
    {                                                                                                   \
        auto late = k_q4k_matvec<LG, R, U, false>;                                                              \
        int grid = persistent_grid(reinterpret_cast<const void *>(late), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                             \
        /* first loads before the dependency wait only when warps have about one task */               \
        const bool early = ntasks * 4 <= static_cast<long long>(grid) * kWarpsPerCta * 5;               \
        auto kern = early ? k_q4k_matvec<LG, R, U, true> : late;                                                 \
        if (early) { /* size through the launched instantiation too (raises its shared-memory limit) */ \
            const int g2 = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
            if (g2 <= 0) return GQ_ERR_SHAPE;                                                           \
            if (g2 < grid) grid = g2;                                                                   \
        }                                                                                               \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, nib, rec, x, y, rows, nsb));        \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

}  // namespace gq
