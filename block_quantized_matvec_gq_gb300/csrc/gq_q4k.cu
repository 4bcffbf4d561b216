// gq_q4k.cu -- Q4_K x f32 decode matvec.
//
// "Metal kernel capability table (Phase B ground truth)", section 1:
// q4k_matvec / q4k_matvec_8sg (144-byte super-blocks, K % 256, rows masked;
// here K % 256 is asserted at dispatch rather than assumed).
//   y_i = sum over super-blocks and sub-blocks s of
//         d*sc_s * sum_j q_j x_j  -  dmin*m_s * sum_j x_j
// The per-32 sums of x are computed once per CTA, inside the staged x blocks.
// The codes enter the FMAs as subnormal floats against x staged with
// per-position power-of-two scales (nib8_sub_fma, stage_x_q4k); every sum is
// scaled by 2^-c until the row result, which is scaled back by 2^c.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U, int kMode>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4k_matvec(const uint4 *__restrict__ nib, const uint4 *__restrict__ rec,
                 const float *__restrict__ x, float *__restrict__ y, int rows, int nsb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    // schedule (chosen by the host): 0 round-robin; 1 balanced; 2 balanced, first loads early
    constexpr bool kBalanced = kMode >= 1, kEarly = kMode == 2;
    __shared__ float part[kWarpsPerCta][kWarpsPerCta * TR];  // tail partial sums [warp][row]
    __shared__ uint32_t red[kWarpsPerCta];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ns = nsb >> 3;
    if constexpr (!kBalanced) {
        // round-robin: task t of the grid goes to warp t % (warps in the grid)
        const int ntasks = (rows + TR - 1) / TR;
        const int first = blockIdx.x * kWarpsPerCta + warp;
        const int stride = gridDim.x * kWarpsPerCta;

        Q4KStream<LG, R, U> st;
        auto setup = [&](int task) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(task * TR + g * R + i, rows - 1);
                st.wp[i] = nib + static_cast<size_t>(r) * nsb + lp;
                st.rp[i] = rec + static_cast<size_t>(r) * ns + (lp >> 3);
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
            /* no early loads in this mode */
        }
        pdl_wait();
        const int c = stage_x_q4k(xs, x, nsb * 32, red);
        pdl_launch_dependents();

        for (int task = first; task < ntasks; task += stride) {
            setup(task);
            // the next task's rows stream into L2 while this one computes
            if (task + stride < ntasks)
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(nib), nsb * 16u,
                                     reinterpret_cast<const uint8_t *>(rec), ns * 16u, (task + stride) * TR, rows, lane);
            float out[R];
            st.run(xs, nsb, lp, out);
            const int r0 = task * TR + g * R;
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + i < rows) y[r0 + i] = scale_pow2(s, c);
            }
        }
    } else {
        const WarpRows cr = warp_rows<TR>(rows, kBalanced, warp);

        Q4KStream<LG, R, U> st;
        // rows r0 + g*R + i of a TR-row task, sub-blocks [blo, bhi) (blo % 8 == 0,
        // so a lane's sub-block position stays lp % 8)
        auto setup = [&](int r0, int blo, int bhi) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(r0 + g * R + i, rows - 1);
                st.wp[i] = nib + static_cast<size_t>(r) * nsb + blo + lp;
                st.rp[i] = rec + static_cast<size_t>(r) * ns + ((blo + lp) >> 3);
            }
            st.prime(bhi - blo, lp);
        };
        // Weights never depend on the previous kernel: prefetch this warp's first
        // rows into L2 before waiting for it and, when warps have about one task
        // each (kEarly, chosen by the host), issue that task's first loads too.
        if (cr.count > 0) {
            const void *rp[TR];
    #pragma unroll
            for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(cr.start + i, rows - 1)) * nsb;
            prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nsb) * 16u, lane);
            if (kEarly) setup(cr.start, 0, nsb);
        }
        pdl_wait();
        const int c = stage_x_q4k(xs, x, nsb * 32, red);
        pdl_launch_dependents();

        for (int j = 0; j < cr.count; ++j) {
            const int r0 = cr.start + j * cr.step;
            if (j > 0 || !kEarly) setup(r0, 0, nsb);
            // the next task's rows stream into L2 while this one computes
            if (j + 1 < cr.count)
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(nib), nsb * 16u,
                                     reinterpret_cast<const uint8_t *>(rec), ns * 16u, r0 + cr.step, rows, lane);
            float out[R];
            st.run(xs, nsb, lp, out);
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + g * R + i < rows) y[r0 + g * R + i] = scale_pow2(s, c);
            }
        }
        if (kBalanced && cr.ntail > 0) {
            int blo, bhi;
            tail_slice(nsb, 8, warp, blo, bhi);
            for (int t0 = 0; t0 < cr.ntail; t0 += TR) {
                setup(cr.tail_begin + t0, blo, bhi);
                float out[R];
                st.run(xs + blo * kXBlk, bhi - blo, lp, out);
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
                y[cr.tail_begin + r] = scale_pow2(s, c);
            }
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
#define CASE(LG, R, U)                                                                                  \
    {                                                                                                   \
        auto rr = k_q4k_matvec<LG, R, U, 0>;                                                                     \
        int grid = persistent_grid(reinterpret_cast<const void *>(rr), kThreadsPerCta, smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                             \
        /* tasks per warp: < 1.75 balanced schedule, <= 1.25 also first loads early */                 \
        const long long w5 = static_cast<long long>(grid) * kWarpsPerCta;                               \
        const int mode = schedule_mode(ntasks, w5, nsb);                                                     \
        auto kern = mode == 2 ? k_q4k_matvec<LG, R, U, 2> : (mode == 1 ? k_q4k_matvec<LG, R, U, 1> : rr);                 \
        if (mode != 0) { /* size through the launched instantiation too (raises its shared-memory limit) */ \
            const int g2 = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
            if (g2 <= 0) return GQ_ERR_SHAPE;                                                           \
            if (g2 < grid) grid = g2;                                                                   \
        }                                                                                               \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, nib, rec, x, y, rows, nsb));       \
    }
    GQ_GEO_SWITCH_R12(geo, CASE);
#undef CASE
}

}  // namespace gq
