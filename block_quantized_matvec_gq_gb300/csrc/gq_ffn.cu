// gq_ffn.cu -- fused gated GELU FFN gate/up pair over Q4_0 weights.
//
// "Gemma 4 M4 Max kernel roadmap", K2 step 5 (gated GELU FFN projection
// pair) and K5 (exact gate/up launch fusion: one pass over x, both weight
// streams); "Metal kernel capability table (Phase B ground truth)",
// section 4 (geglu_gelu_tanh with the +-15 clamp; finding F1 is the NaN of
// an unclamped fused variant).
//   h_i = gelu_tanh(W_gate[i] . x) * (W_up[i] . x)
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U, int kMode>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_ffn_gate_up(const uint4 *__restrict__ gnib, const uint16_t *__restrict__ gsc,
                  const uint4 *__restrict__ unib, const uint16_t *__restrict__ usc,
                  const float *__restrict__ x, float *__restrict__ h, int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    // schedule (chosen by the host): 0 round-robin; 1 balanced; 2 balanced, first loads early
    constexpr bool kBalanced = kMode >= 1, kEarly = kMode == 2;
    __shared__ float gpart[kWarpsPerCta][kWarpsPerCta * TR];  // tail partial sums [warp][row]
    __shared__ float upart[kWarpsPerCta][kWarpsPerCta * TR];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    if constexpr (!kBalanced) {
        // round-robin: task t of the grid goes to warp t % (warps in the grid)
        const int ntasks = (rows + TR - 1) / TR;
        const int first = blockIdx.x * kWarpsPerCta + warp;
        const int stride = gridDim.x * kWarpsPerCta;

        // rows 0..R-1 of the stream are gate rows, R..2R-1 the matching up rows
        Q40Stream<LG, 2 * R, U> st;
        auto setup = [&](int task) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(task * TR + g * R + i, rows - 1);
                st.wp[i] = gnib + static_cast<size_t>(r) * nb + lp;
                st.sp[i] = gsc + static_cast<size_t>(r) * nb + lp;
                st.wp[R + i] = unib + static_cast<size_t>(r) * nb + lp;
                st.sp[R + i] = usc + static_cast<size_t>(r) * nb + lp;
            }
            st.prime(nb, lp);
        };
        // Weights never depend on the previous kernel: prefetch this warp's first
        // rows into L2 before waiting for it and, when warps have about one task
        // each (kEarly, chosen by the host), issue that task's first loads too.
        // (Measured: with several tasks per warp the early loads cost more than
        // they save.)
        if (first < ntasks) {
            const void *rp[2 * TR];
    #pragma unroll
            for (int i = 0; i < TR; ++i) {
                const size_t r = static_cast<size_t>(min(first * TR + i, rows - 1));
                rp[i] = gnib + r * nb;
                rp[TR + i] = unib + r * nb;
            }
            prefetch_rows_l2<2 * TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
            /* no early loads in this mode */
        }
        pdl_wait();
        stage_x_q4<false>(xs, x, nb * 32);
        pdl_launch_dependents();

        for (int task = first; task < ntasks; task += stride) {
            setup(task);
            // the next task's rows stream into L2 while this one computes
            if (task + stride < ntasks) {
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(gnib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(gsc), nb * 2u, (task + stride) * TR, rows, lane);
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(unib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(usc), nb * 2u, (task + stride) * TR, rows, lane);
            }
            float out[2 * R];
            st.run(xs, nb, lp, out);
            const int r0 = task * TR + g * R;
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float gv = group_sum<LG>(out[i]);
                const float uv = group_sum<LG>(out[R + i]);
                if (lp == 0 && r0 + i < rows) h[r0 + i] = gelu_tanh(gv) * uv;
            }
        }
    } else {
        const WarpRows cr = warp_rows<TR>(rows, kBalanced, warp);

        // rows 0..R-1 of the stream are gate rows, R..2R-1 the matching up rows
        Q40Stream<LG, 2 * R, U> st;
        auto setup = [&](int r0, int blo, int bhi) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(r0 + g * R + i, rows - 1);
                st.wp[i] = gnib + static_cast<size_t>(r) * nb + blo + lp;
                st.sp[i] = gsc + static_cast<size_t>(r) * nb + blo + lp;
                st.wp[R + i] = unib + static_cast<size_t>(r) * nb + blo + lp;
                st.sp[R + i] = usc + static_cast<size_t>(r) * nb + blo + lp;
            }
            st.prime(bhi - blo, lp);
        };
        // Weights never depend on the previous kernel: prefetch this warp's first
        // rows into L2 before waiting for it and, when warps have about one task
        // each (kEarly, chosen by the host), issue that task's first loads too.
        if (cr.count > 0) {
            const void *rp[2 * TR];
    #pragma unroll
            for (int i = 0; i < TR; ++i) {
                const size_t r = static_cast<size_t>(min(cr.start + i, rows - 1));
                rp[i] = gnib + r * nb;
                rp[TR + i] = unib + r * nb;
            }
            prefetch_rows_l2<2 * TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
            if (kEarly) setup(cr.start, 0, nb);
        }
        pdl_wait();
        stage_x_q4<false>(xs, x, nb * 32);
        pdl_launch_dependents();

        for (int j = 0; j < cr.count; ++j) {
            const int r0 = cr.start + j * cr.step;
            if (j > 0 || !kEarly) setup(r0, 0, nb);
            // the next task's rows stream into L2 while this one computes
            if (j + 1 < cr.count) {
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(gnib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(gsc), nb * 2u, r0 + cr.step, rows, lane);
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(unib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(usc), nb * 2u, r0 + cr.step, rows, lane);
            }
            float out[2 * R];
            st.run(xs, nb, lp, out);
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float gv = group_sum<LG>(out[i]);
                const float uv = group_sum<LG>(out[R + i]);
                if (lp == 0 && r0 + g * R + i < rows) h[r0 + g * R + i] = gelu_tanh(gv) * uv;
            }
        }
        if (kBalanced && cr.ntail > 0) {
            int blo, bhi;
            tail_slice(nb, 1, warp, blo, bhi);
            for (int t0 = 0; t0 < cr.ntail; t0 += TR) {
                setup(cr.tail_begin + t0, blo, bhi);
                float out[2 * R];
                st.run(xs + blo * kXBlk, bhi - blo, lp, out);
    #pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float gv = group_sum<LG>(out[i]);
                    const float uv = group_sum<LG>(out[R + i]);
                    if (lp == 0) {
                        gpart[warp][t0 + g * R + i] = gv;
                        upart[warp][t0 + g * R + i] = uv;
                    }
                }
            }
            __syncthreads();
            for (int r = threadIdx.x; r < cr.ntail; r += kThreadsPerCta) {
                float gv = 0.f, uv = 0.f;
    #pragma unroll
                for (int w = 0; w < kWarpsPerCta; ++w) {
                    gv += gpart[w][r];
                    uv += upart[w][r];
                }
                h[cr.tail_begin + r] = gelu_tanh(gv) * uv;
            }
        }
    }
}

int launch_ffn_gate_up(const void *Wg, const void *Wu, const float *x, float *h, int rows, int K,
                       MatvecGeo geo, cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *gn = static_cast<const uint4 *>(Wg);
    const uint16_t *gs = reinterpret_cast<const uint16_t *>(gn + static_cast<size_t>(rows) * nb);
    const uint4 *un = static_cast<const uint4 *>(Wu);
    const uint16_t *us = reinterpret_cast<const uint16_t *>(un + static_cast<size_t>(rows) * nb);
    const size_t smem = static_cast<size_t>(nb) * kXBlk * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                  \
    {                                                                                                   \
        auto rr = k_ffn_gate_up<LG, R, U, 0>;                                                                     \
        int grid = persistent_grid(reinterpret_cast<const void *>(rr), kThreadsPerCta, smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                             \
        /* tasks per warp: < 1.75 balanced schedule, <= 1.25 also first loads early */                 \
        const long long w5 = static_cast<long long>(grid) * kWarpsPerCta;                               \
        const int mode = schedule_mode(ntasks, w5, nb);                                                     \
        auto kern = mode == 2 ? k_ffn_gate_up<LG, R, U, 2> : (mode == 1 ? k_ffn_gate_up<LG, R, U, 1> : rr);                 \
        if (mode != 0) { /* size through the launched instantiation too (raises its shared-memory limit) */ \
            const int g2 = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
            if (g2 <= 0) return GQ_ERR_SHAPE;                                                           \
            if (g2 < grid) grid = g2;                                                                   \
        }                                                                                               \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, gn, gs, un, us, x, h, rows, nb));       \
    }
    GQ_GEO_SWITCH_R12(geo, CASE);
#undef CASE
}

}  // namespace gq
