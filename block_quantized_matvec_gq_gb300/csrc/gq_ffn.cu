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

template <int LG, int R, int U, int P>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_ffn_gate_up(const uint4 *__restrict__ gnib, const uint16_t *__restrict__ gsc,
                  const uint4 *__restrict__ unib, const uint16_t *__restrict__ usc,
                  const float *__restrict__ x, float *__restrict__ h, int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const int first = blockIdx.x * kWarpsPerCta + warp;

    if (first < ntasks) {
        const void *rp[2 * TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) {
            const size_t r = static_cast<size_t>(min(first * TR + i, rows - 1));
            rp[i] = gnib + r * nb;
            rp[TR + i] = unib + r * nb;
        }
        prefetch_rows_l2<2 * TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
    }
    pdl_wait();
    stage_x_perm8(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += gridDim.x * kWarpsPerCta) {
        const int r0 = task * TR + g * R;
        const uint4 *wp[2 * R];
        const uint16_t *sp[2 * R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(r0 + i, rows - 1);
            wp[i] = gnib + static_cast<size_t>(r) * nb;
            sp[i] = gsc + static_cast<size_t>(r) * nb;
            wp[R + i] = unib + static_cast<size_t>(r) * nb;
            sp[R + i] = usc + static_cast<size_t>(r) * nb;
        }
        float out[2 * R];
        if (P == 2)
            q4_0_stream2<LG, 2 * R, U>(wp, sp, xs, nb, lp, out);
        else
            q4_0_stream<LG, 2 * R, U>(wp, sp, xs, nb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float gv = group_sum<LG>(out[i]);
            const float uv = group_sum<LG>(out[R + i]);
            if (lp == 0 && r0 + i < rows) h[r0 + i] = gelu_tanh(gv) * uv;
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
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                 \
    {                                                                                                  \
        auto kern = k_ffn_gate_up<LG, R, U, PP>;                                                       \
        const int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                            \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, gn, gs, un, us, x, h, rows, nb)); \
    }
    if (geo.p == 2) {
        constexpr int PP = 2;
        GQ_PAIR_SWITCH(geo, CASE);
    } else {
        constexpr int PP = 1;
        GQ_GEO_SWITCH_R12(geo, CASE);
    }
#undef CASE
}

}  // namespace gq
