// gq_matvec.cu -- decode matvec kernels (Q4_0, Q8_0, Q4_K), the fused gated
// GELU gate/up pair, and the Q8_0 tied-logit projection with soft-cap and
// top-k.
//
// "Gemma 4 M4 Max kernel roadmap", K2 "Metal decode path": step 1 (direct
// Q4_0 matrix-vector with fused dequantization and F32 accumulation), step 5
// (gated GELU FFN projection pair), step 6 (Q8_0 output projection and
// on-GPU top-k); K5 (pair-valued (value, token) frontiers merged level by
// level).  "Metal kernel capability table (Phase B ground truth)", section 1
// (q4_f32_matvec, q4k_matvec: rows masked; here K is never truncated) and
// section 4 (GELU-tanh with the +-15 clamp, finding F1).
//
// Every kernel is persistent (grid = SMs x resident CTAs, capped by the
// work), stages x once per CTA into shared memory with cp.async, and then
// streams its share of weight rows with 16-byte evict-first loads.
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

constexpr int kThreadsPerCta = 256;
constexpr int kWarpsPerCta = kThreadsPerCta / 32;

// ================================================================ kernels

template <int LG, int R, int U>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q4_0_matvec(const uint4 *__restrict__ nib, const uint16_t *__restrict__ dsc,
                  const float *__restrict__ x, float *__restrict__ y, int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;

    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = blockIdx.x * kWarpsPerCta + warp; task < ntasks; task += gridDim.x * kWarpsPerCta) {
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
        q4_0_stream<LG, R, U>(wp, sp, xs, nb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(out[i]);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

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

    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = blockIdx.x * kWarpsPerCta + warp; task < ntasks; task += gridDim.x * kWarpsPerCta) {
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

// Per-block sums of x (for the Q4_K min term), after stage_x.
__device__ __forceinline__ void stage_xsum(float *xsum, const float *xs, int nb)
{
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float4 v = ld_xchunk(xs, b, m);
            s += v.x;
            s += v.y;
            s += v.z;
            s += v.w;
        }
        xsum[b] = s;
    }
    __syncthreads();
}

template <int LG, int R, int U>
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

    pdl_wait();
    stage_x(xs, x, nsb * 32);
    stage_xsum(xsum, xs, nsb);
    pdl_launch_dependents();

    for (int task = blockIdx.x * kWarpsPerCta + warp; task < ntasks; task += gridDim.x * kWarpsPerCta) {
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
        q4k_stream<LG, R, U>(wp, rp, xs, xsum, nsb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float s = group_sum<LG>(out[i]);
            if (lp == 0 && r0 + i < rows) y[r0 + i] = s;
        }
    }
}

// GELU, tanh form, with the tanh argument clamped to +-15 (tanh(15) rounds
// to 1 in f32, so the clamp changes no finite result and keeps it finite).
__device__ __forceinline__ float gelu_tanh(float a)
{
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    float t = k0 * (a + 0.044715f * a * a * a);
    t = fminf(fmaxf(t, -15.f), 15.f);
    return 0.5f * a * (1.f + tanhf(t));
}

template <int LG, int R, int U>
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

    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    for (int task = blockIdx.x * kWarpsPerCta + warp; task < ntasks; task += gridDim.x * kWarpsPerCta) {
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
        q4_0_stream<LG, 2 * R, U>(wp, sp, xs, nb, lp, out);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float gv = group_sum<LG>(out[i]);
            const float uv = group_sum<LG>(out[R + i]);
            if (lp == 0 && r0 + i < rows) h[r0 + i] = gelu_tanh(gv) * uv;
        }
    }
}

// ---------------------------------------------------------------- logits + top-k
// Phase 1: every warp streams its rows, soft-caps each logit, optionally
// stores it, and keeps the k best (value, row) keys of the rows it has seen
// in a warp-resident sorted list; at the end the CTA merges its warps' lists
// and writes k keys to the workspace.
template <int LG, int R, int U>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q8_0_logits_topk(const uint4 *__restrict__ qb, const uint16_t *__restrict__ dsc,
                       const float *__restrict__ x, float softcap, int k,
                       float *__restrict__ logits, unsigned long long *__restrict__ ws, int rows,
                       int nb)
{
    extern __shared__ __align__(16) float xs[];
    __shared__ unsigned long long cta_keys[kWarpsPerCta * GQ_MAX_TOPK];
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const bool cap = softcap > 0.f;

    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    WarpTopK top;
    top.init();
    unsigned long long thr = 0ull;

    for (int task = blockIdx.x * kWarpsPerCta + warp; task < ntasks; task += gridDim.x * kWarpsPerCta) {
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
            float l = group_sum<LG>(out[i]);
            const int r = r0 + i;
            if (cap) l = softcap * tanhf(__fdiv_rn(l, softcap));
            if (lp == 0 && r < rows && logits != nullptr) logits[r] = l;
            const unsigned long long key = (lp == 0 && r < rows) ? topk_key(l, static_cast<uint32_t>(r)) : 0ull;
            unsigned int want = __ballot_sync(0xffffffffu, key > thr);
            while (want) {
                const int src = __ffs(want) - 1;
                want &= want - 1;
                const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
                if (kk > thr) {
                    top.insert(kk, k);
                    thr = top.kth(k);
                }
            }
        }
    }

    // merge the warps' lists (lane j holds entry j in e0 and entry j+32 in e1)
    for (int j = lane; j < k; j += 32) cta_keys[warp * k + j] = (j < 32) ? top.e0 : top.e1;
    __syncthreads();
    if (warp == 0) {
        top.init();
        thr = 0ull;
        for (int base = 0; base < kWarpsPerCta * k; base += 32) {
            const int j = base + lane;
            const unsigned long long key = (j < kWarpsPerCta * k) ? cta_keys[j] : 0ull;
            unsigned int want = __ballot_sync(0xffffffffu, key > thr);
            while (want) {
                const int src = __ffs(want) - 1;
                want &= want - 1;
                const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
                if (kk > thr) {
                    top.insert(kk, k);
                    thr = top.kth(k);
                }
            }
        }
        if (lane < k) ws[static_cast<size_t>(blockIdx.x) * k + lane] = top.e0;
        if (lane + 32 < k) ws[static_cast<size_t>(blockIdx.x) * k + lane + 32] = top.e1;
    }
}

// Phase 2: one CTA merges the n per-CTA lists (n*k keys) into the final k.
constexpr int kMergeThreads = 1024;
__global__ void __launch_bounds__(kMergeThreads)
    k_topk_merge(const unsigned long long *__restrict__ ws, int nkeys, int k, int *__restrict__ idx,
                 float *__restrict__ val)
{
    __shared__ unsigned long long wkeys[(kMergeThreads / 32) * GQ_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nwarps = kMergeThreads / 32;
    pdl_wait();
    WarpTopK top;
    top.init();
    unsigned long long thr = 0ull;
    // each warp takes a contiguous slice of the keys
    const int per = (nkeys + nwarps - 1) / nwarps;
    const int lo = warp * per, hi = min(nkeys, lo + per);
    for (int base = lo; base < hi; base += 32) {
        const int j = base + lane;
        const unsigned long long key = (j < hi) ? ws[j] : 0ull;
        unsigned int want = __ballot_sync(0xffffffffu, key > thr);
        while (want) {
            const int src = __ffs(want) - 1;
            want &= want - 1;
            const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
            if (kk > thr) {
                top.insert(kk, k);
                thr = top.kth(k);
            }
        }
    }
    if (lane < k) wkeys[warp * k + lane] = top.e0;
    if (lane + 32 < k) wkeys[warp * k + lane + 32] = top.e1;
    __syncthreads();
    if (warp == 0) {
        top.init();
        thr = 0ull;
        for (int base = 0; base < nwarps * k; base += 32) {
            const int j = base + lane;
            const unsigned long long key = (j < nwarps * k) ? wkeys[j] : 0ull;
            unsigned int want = __ballot_sync(0xffffffffu, key > thr);
            while (want) {
                const int src = __ffs(want) - 1;
                want &= want - 1;
                const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
                if (kk > thr) {
                    top.insert(kk, k);
                    thr = top.kth(k);
                }
            }
        }
        if (lane < k) {
            idx[lane] = static_cast<int>(key_row(top.e0));
            val[lane] = key_value(top.e0);
        }
        if (lane + 32 < k) {
            idx[lane + 32] = static_cast<int>(key_row(top.e1));
            val[lane + 32] = key_value(top.e1);
        }
    }
}

// ================================================================ launchers

MatvecGeo choose_matvec_geo(int format, int rows, int nb)
{
    // Lane-group width: the widest of 32/16/8 that divides the blocks per row
    // (no idle lanes at the row tail); 32 when none does (tail masked).
    int lg = (nb % 32 == 0) ? 32 : (nb % 16 == 0) ? 16 : (nb % 8 == 0) ? 8 : 32;
    // Rows per lane group: enough x reuse (G*R >= 4 rows share one x load),
    // and enough warp tasks to fill the GPU.
    const int G = 32 / lg;
    int r = (G >= 2) ? 2 : 4;
    const int warps_wanted = sm_count() * 16;
    if (r == 4 && (rows + G * 4 - 1) / (G * 4) < warps_wanted) r = 2;
    (void)format;
    return MatvecGeo{lg, r, 2, kWarpsPerCta};
}

static int grid_for(const void *kern, size_t smem, int ntasks)
{
    const int occ = ctas_per_sm(kern, kThreadsPerCta, smem);
    if (occ <= 0) return -1;
    const int want = (ntasks + kWarpsPerCta - 1) / kWarpsPerCta;
    const int cap = sm_count() * occ;
    return want < cap ? want : cap;
}

#define GQ_GEO_SWITCH(geo, CASE)                                   \
    do {                                                            \
        if ((geo).u != 2) return GQ_ERR_SHAPE;                      \
        if ((geo).lg == 32 && (geo).r == 2) { CASE(32, 2, 2); }     \
        else if ((geo).lg == 32 && (geo).r == 4) { CASE(32, 4, 2); } \
        else if ((geo).lg == 16 && (geo).r == 2) { CASE(16, 2, 2); } \
        else if ((geo).lg == 16 && (geo).r == 4) { CASE(16, 4, 2); } \
        else if ((geo).lg == 8 && (geo).r == 2) { CASE(8, 2, 2); }   \
        else if ((geo).lg == 8 && (geo).r == 4) { CASE(8, 4, 2); }   \
        else if ((geo).lg == 8 && (geo).r == 1) { CASE(8, 1, 2); }   \
        else if ((geo).lg == 16 && (geo).r == 1) { CASE(16, 1, 2); } \
        else if ((geo).lg == 32 && (geo).r == 1) { CASE(32, 1, 2); } \
        else return GQ_ERR_SHAPE;                                   \
    } while (0)

int launch_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const int TR = (32 / geo.lg) * geo.r;
    const int ntasks = (rows + TR - 1) / TR;
#define CASE(LG, R, U)                                                                  \
    {                                                                                   \
        auto kern = k_q4_0_matvec<LG, R, U>;                                            \
        const int grid = grid_for(reinterpret_cast<const void *>(kern), smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                             \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, \
                                      nib, dsc, x, y, rows, nb));                       \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

int launch_q8_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *qb = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(qb + static_cast<size_t>(rows) * nb * 2);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const int TR = (32 / geo.lg) * geo.r;
    const int ntasks = (rows + TR - 1) / TR;
#define CASE(LG, R, U)                                                                  \
    {                                                                                   \
        auto kern = k_q8_0_matvec<LG, R, U>;                                            \
        const int grid = grid_for(reinterpret_cast<const void *>(kern), smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                             \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, \
                                      qb, dsc, x, y, rows, nb));                        \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

int launch_q4k_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo geo,
                      cudaStream_t s)
{
    const int nsb = K / 32, ns = K / 256;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint4 *rec = nib + static_cast<size_t>(rows) * nsb;
    const size_t smem = static_cast<size_t>(K) * sizeof(float) + static_cast<size_t>(nsb) * sizeof(float);
    const int TR = (32 / geo.lg) * geo.r;
    const int ntasks = (rows + TR - 1) / TR;
    (void)ns;
#define CASE(LG, R, U)                                                                  \
    {                                                                                   \
        auto kern = k_q4k_matvec<LG, R, U>;                                             \
        const int grid = grid_for(reinterpret_cast<const void *>(kern), smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                             \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, \
                                      nib, rec, x, y, rows, nsb));                      \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
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
    const int TR = (32 / geo.lg) * geo.r;
    const int ntasks = (rows + TR - 1) / TR;
#define CASE(LG, R, U)                                                                  \
    {                                                                                   \
        auto kern = k_ffn_gate_up<LG, R, U>;                                            \
        const int grid = grid_for(reinterpret_cast<const void *>(kern), smem, ntasks);  \
        if (grid <= 0) return GQ_ERR_SHAPE;                                             \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, \
                                      gn, gs, un, us, x, h, rows, nb));                 \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

// Upper bound on the CTAs of the logits kernel, fixed so the workspace size
// depends only on the arguments, not on the GPU.
constexpr int kLogitsMaxCtas = 2048;

size_t logits_topk_ws_bytes(int rows, int K, int k)
{
    (void)K;
    const long long tasks_ctas = (static_cast<long long>(rows) + 7) / 8;
    const long long ctas = tasks_ctas < kLogitsMaxCtas ? tasks_ctas : kLogitsMaxCtas;
    return static_cast<size_t>(ctas) * static_cast<size_t>(k) * sizeof(unsigned long long);
}

int launch_logits_topk(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                       float *logits, void *ws, size_t ws_bytes, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *qb = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(qb + static_cast<size_t>(rows) * nb * 2);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const int TR = (32 / geo.lg) * geo.r;
    const int ntasks = (rows + TR - 1) / TR;
    unsigned long long *keys = static_cast<unsigned long long *>(ws);
#define CASE(LG, R, U)                                                                           \
    {                                                                                            \
        auto kern = k_q8_0_logits_topk<LG, R, U>;                                                \
        int grid = grid_for(reinterpret_cast<const void *>(kern), smem, ntasks);                 \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                      \
        if (grid > kLogitsMaxCtas) grid = kLogitsMaxCtas;                                        \
        if (static_cast<size_t>(grid) * k * sizeof(unsigned long long) > ws_bytes)               \
            return GQ_ERR_WORKSPACE;                                                             \
        cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, qb, dsc, x,  \
                                   softcap, k, logits, keys, rows, nb);                          \
        if (e != cudaSuccess) return GQ_ERR_CUDA;                                                \
        e = launch_pdl(k_topk_merge, dim3(1), dim3(kMergeThreads), 0, s,                         \
                       static_cast<const unsigned long long *>(keys), grid * k, k, idx, val);    \
        return status_from(e);                                                                   \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

}  // namespace gq
