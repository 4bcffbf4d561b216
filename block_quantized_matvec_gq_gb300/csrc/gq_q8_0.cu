// gq_q8_0.cu -- Q8_0 x f32 decode matvec.
//
// "Gemma 4 M4 Max kernel roadmap", K2 step 6 (the Q8_0 embedding/output
// projection; its top-k form is gq_logits.cu).  "Metal kernel capability
// table (Phase B ground truth)", section 1, q8_matvec (here the fp16 scale
// stays with its block, in the packed scale plane).
//
// Each lane loads a whole 32-byte block of offset-binary codes per row with
// one 256-bit load; codes become exact f32 through PRMT + one FADD.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

template <int LG, int R, int U>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q8_0_matvec(const uint4 *__restrict__ qb, const uint16_t *__restrict__ dsc,
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
        for (int i = 0; i < TR; ++i) rp[i] = qb + static_cast<size_t>(min(first * TR + i, rows - 1)) * nb * 2;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nb) * 32u, lane);
    }
    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = first; task < ntasks; task += gridDim.x * kWarpsPerCta) {
        const int r0 = task * TR + g * R;
        const uint4 *wp[R];
        const uint16_t *sp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(r0 + i, rows - 1);
            wp[i] = qb + static_cast<size_t>(r) * nb * 2;
            sp[i] = dsc + static_cast<size_t>(r) * nb;
        }
        float out[R];
        q8_0_stream<LG, R, U>(wp, sp, xs, nb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(out[i]);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

int launch_q8_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *qb = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(qb + static_cast<size_t>(rows) * nb * 2);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                 \
    {                                                                                                  \
        auto kern = k_q8_0_matvec<LG, R, U>;                                                           \
        const int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                            \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, qb, dsc, x, y, rows, nb)); \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

}  // namespace gq
