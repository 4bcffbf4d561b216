// gq_q4_0.cu -- Q4_0 x f32 decode matvec.
//
// "Gemma 4 M4 Max kernel roadmap", K2 "Metal decode path", step 1: direct
// Q4_0 matrix-vector product with fused dequantization and F32
// accumulation.  "Metal kernel capability table (Phase B ground truth)",
// section 1, q4_f32_matvec (rows masked; here K is never truncated).
//
// Persistent kernel: each CTA stages its input vector once (padded 144-byte
// blocks), then its warps stream packed Q4_0 rows (16-byte nibble loads +
// fp16 scales); see gq_matvec.cuh for the lane geometry and the exact
// nibble-to-f32 step.
//
// The input vector is x itself, or -- the down projection of a gated GELU
// FFN with the gate applied while the input is read ("Metal kernel
// capability table (Phase B ground truth)", section 4, the fused GELU-tanh
// down kernels that take the gate and up vectors) -- h = gelu_tanh(g) * u,
// formed in f32 as the vector is staged, with the tanh argument clamped to
// +-15 (finding F1: the pages' fused kernels lacked the clamp their
// separated twins carry, and gave NaN for large gate values).
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

// Input: x.
struct InX {
    const float *__restrict__ x;
    __device__ __forceinline__ void stage(float *xs, int K) const { stage_x_q4<false>(xs, x, K); }
};

// Input: gelu_tanh(g) * u, in the staged layout of stage_x_q4 (8-element
// group i at block i / 4, offset 8 (i % 4), as elements 0,4,1,5 | 2,6,3,7).
// All threads of the CTA take part; ends with a CTA barrier.
struct InGeglu {
    const float *__restrict__ g;
    const float *__restrict__ u;
    __device__ __forceinline__ void stage(float *xs, int K) const
    {
        for (int i = threadIdx.x; i < (K >> 3); i += blockDim.x) {
            const float4 g0 = *reinterpret_cast<const float4 *>(g + 8 * i);
            const float4 g1 = *reinterpret_cast<const float4 *>(g + 8 * i + 4);
            const float4 u0 = *reinterpret_cast<const float4 *>(u + 8 * i);
            const float4 u1 = *reinterpret_cast<const float4 *>(u + 8 * i + 4);
            const float4 a = make_float4(gelu_tanh(g0.x) * u0.x, gelu_tanh(g0.y) * u0.y, gelu_tanh(g0.z) * u0.z,
                                         gelu_tanh(g0.w) * u0.w);
            const float4 b = make_float4(gelu_tanh(g1.x) * u1.x, gelu_tanh(g1.y) * u1.y, gelu_tanh(g1.z) * u1.z,
                                         gelu_tanh(g1.w) * u1.w);
            float *dst = xs + (i >> 2) * kXBlk + 8 * (i & 3);
            *reinterpret_cast<float4 *>(dst) = make_float4(a.x, b.x, a.y, b.y);
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(a.z, b.z, a.w, b.w);
        }
        __syncthreads();
    }
};

template <int LG, int R, int U, int kMode, class In>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4_0_matvec(const uint4 *__restrict__ nib, const uint16_t *__restrict__ dsc, In in, float *__restrict__ y,
                  int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    // schedule (chosen by the host): 0 round-robin; 1 balanced; 2 balanced, first loads early
    constexpr bool kBalanced = kMode >= 1, kEarly = kMode == 2;
    __shared__ float part[kWarpsPerCta][kWarpsPerCta * TR];  // tail partial sums [warp][row]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    if constexpr (!kBalanced) {
        // round-robin: task t of the grid goes to warp t % (warps in the grid)
        const int ntasks = (rows + TR - 1) / TR;
        const int first = blockIdx.x * kWarpsPerCta + warp;
        const int stride = gridDim.x * kWarpsPerCta;

        Q40Stream<LG, R, U> st;
        auto setup = [&](int task) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(task * TR + g * R + i, rows - 1);
                st.wp[i] = nib + static_cast<size_t>(r) * nb + lp;
                st.sp[i] = dsc + static_cast<size_t>(r) * nb + lp;
            }
            st.prime(nb, lp);
        };
        // Weights never depend on the previous kernel: prefetch this warp's first
        // rows into L2 before waiting for it and, when warps have about one task
        // each (kEarly, chosen by the host), issue that task's first loads too.
        // (Measured: with several tasks per warp the early loads cost more than
        // they save.)
        if (first < ntasks) {
            const void *rp[TR];
    #pragma unroll
            for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(first * TR + i, rows - 1)) * nb;
            prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
            /* no early loads in this mode */
        }
        pdl_wait();
        in.stage(xs, nb * 32);
        pdl_launch_dependents();

        for (int task = first; task < ntasks; task += stride) {
            setup(task);
            // the next task's rows stream into L2 while this one computes
            if (task + stride < ntasks)
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(nib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(dsc), nb * 2u, (task + stride) * TR, rows, lane);
            float out[R];
            st.run(xs, nb, lp, out);
            const int r0 = task * TR + g * R;
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
            }
        }
    } else {
        const WarpRows cr = warp_rows<TR>(rows, kBalanced, warp);

        Q40Stream<LG, R, U> st;
        // rows r0 + g*R + i of a TR-row task, blocks [blo, bhi)
        auto setup = [&](int r0, int blo, int bhi) {
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = min(r0 + g * R + i, rows - 1);
                st.wp[i] = nib + static_cast<size_t>(r) * nb + blo + lp;
                st.sp[i] = dsc + static_cast<size_t>(r) * nb + blo + lp;
            }
            st.prime(bhi - blo, lp);
        };
        // Weights never depend on the previous kernel: prefetch this warp's first
        // rows into L2 before waiting for it and, when warps have about one task
        // each (kEarly, chosen by the host), issue that task's first loads too.
        // (Measured: with several tasks per warp the early loads cost more than
        // they save.)
        if (cr.count > 0) {
            const void *rp[TR];
    #pragma unroll
            for (int i = 0; i < TR; ++i) rp[i] = nib + static_cast<size_t>(min(cr.start + i, rows - 1)) * nb;
            prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nb) * 16u, lane);
            if (kEarly) setup(cr.start, 0, nb);
        }
        pdl_wait();
        in.stage(xs, nb * 32);
        pdl_launch_dependents();

        for (int j = 0; j < cr.count; ++j) {
            const int r0 = cr.start + j * cr.step;
            if (j > 0 || !kEarly) setup(r0, 0, nb);
            // the next task's rows stream into L2 while this one computes
            if (j + 1 < cr.count)
                prefetch_task_l2<TR>(reinterpret_cast<const uint8_t *>(nib), nb * 16u,
                                     reinterpret_cast<const uint8_t *>(dsc), nb * 2u, r0 + cr.step, rows, lane);
            float out[R];
            st.run(xs, nb, lp, out);
    #pragma unroll
            for (int i = 0; i < R; ++i) {
                const float s = group_sum<LG>(out[i]);
                if (lp == 0 && r0 + g * R + i < rows) y[r0 + g * R + i] = s;
            }
        }
        if (kBalanced && cr.ntail > 0) {
            int blo, bhi;
            tail_slice(nb, 1, warp, blo, bhi);
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
                y[cr.tail_begin + r] = s;
            }
        }
    }
}

template <class In>
static int launch_q4_0(const void *W, In in, float *y, int rows, int K, MatvecGeo geo, cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb);
    const size_t smem = static_cast<size_t>(nb) * kXBlk * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
#define CASE(LG, R, U)                                                                                  \
    {                                                                                                   \
        auto rr = k_q4_0_matvec<LG, R, U, 0, In>;                                                                     \
        int grid = persistent_grid(reinterpret_cast<const void *>(rr), kThreadsPerCta, smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                             \
        /* tasks per warp: < 1.75 balanced schedule, <= 1.25 also first loads early */                 \
        const long long w5 = static_cast<long long>(grid) * kWarpsPerCta;                               \
        const int mode = schedule_mode(ntasks, w5, nb);                                                     \
        auto kern = mode == 2 ? k_q4_0_matvec<LG, R, U, 2, In> : (mode == 1 ? k_q4_0_matvec<LG, R, U, 1, In> : rr);                 \
        if (mode != 0) { /* size through the launched instantiation too (raises its shared-memory limit) */ \
            const int g2 = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
            if (g2 <= 0) return GQ_ERR_SHAPE;                                                           \
            if (g2 < grid) grid = g2;                                                                   \
        }                                                                                               \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, nib, dsc, in, y, rows, nb));       \
    }
    GQ_GEO_SWITCH_R12(geo, CASE);
#undef CASE
}

int launch_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo, cudaStream_t s)
{
    return launch_q4_0(W, InX{x}, y, rows, K, geo, s);
}

int launch_q4_0_geglu_down(const void *W, const float *g, const float *u, float *y, int rows, int K, MatvecGeo geo,
                           cudaStream_t s)
{
    return launch_q4_0(W, InGeglu{g, u}, y, rows, K, geo, s);
}

}  // namespace gq
