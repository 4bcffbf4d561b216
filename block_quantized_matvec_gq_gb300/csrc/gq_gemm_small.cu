// gq_gemm_small.cu -- the Q4_0 x Q8_0 contraction for small token batches
// (M <= 24 in passes of up to 8 tokens: a verifier's few tokens, a short
// prompt), on the CUDA cores.
//
// "Gemma 4 M4 Max kernel roadmap", K3 "prefill path" (batched Q4_0 kernels;
// the fixed-eight verifier and the 32-prompt tile sit between decode and the
// 512-token prefill):
//   D[t][r][b] = sum_{j<32} Xq[t][32b+j] * (q_w[r][32b+j] - 8)   (int32, exact)
//   Y[t][r]    = sum_b d_w[r][b] * dx[t][b] * D[t][r][b]          (f32)
//
// With few tokens the tensor-core tiles (128 tokens) are mostly padding and
// the weight-piece conversion dominates; here every weight is decoded once
// and applied to all M tokens, like the decode matvec:
// * each CTA stages the codes of all (up to MT) tokens in shared memory once:
//   per (token, block) 48 bytes = the 32 codes as 8 words in the order the
//   nibble unpacking below produces (elements 0,2,4,6 | 1,3,5,7 of each
//   8-element group), the block's code sum, padding (16-byte aligned, and a
//   48-byte stride keeps the 16-byte loads of 8 consecutive lanes on distinct
//   banks); and dx of every (token, block);
// * a warp takes two rows; lane l takes blocks l, l + 32, ... of both rows
//   (16-byte coalesced nibble loads), unpacks each nibble word into two words
//   of bytes q in [0, 15], and for every token forms the exact block dot as
//   8 __dp4a of q with the codes minus 8 * (code sum), then folds
//   (d_w * dx) * D into that token's f32 accumulator;
// * the 32 lanes' partial sums are added by a butterfly, and lane t writes
//   token t's output.
// Tokens past M are staged as zeros (their D and dx are 0); they are never
// stored.  Rows past the end are skipped.
#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {
namespace small {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kXW = 12;  // words per (token, block) in shared memory: 8 codes, 1 sum, 3 pad

template <int MT>
__global__ void __launch_bounds__(kThreads)
    k_gemm_small(const uint4 *__restrict__ nib, const uint16_t *__restrict__ dsc, const int8_t *__restrict__ Xq,
                 const float *__restrict__ dx, float *__restrict__ Y, int rows, int nb, int M)
{
    extern __shared__ __align__(16) uint32_t sm[];
    uint32_t *sx = sm;                                                   // [MT][nb][kXW]
    float *sdx = reinterpret_cast<float *>(sm + static_cast<size_t>(MT) * nb * kXW);  // [MT][nb]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_launch_dependents();
    pdl_wait();
    // ---- stage the codes, their block sums and the scales of all tokens
    for (int i = threadIdx.x; i < MT * nb; i += kThreads) {
        const int t = i / nb, b = i - t * nb;
        uint32_t *dst = sx + static_cast<size_t>(i) * kXW;
        if (t < M) {
            const uint4 *src = reinterpret_cast<const uint4 *>(Xq + (static_cast<size_t>(t) * nb + b) * 32);
            const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            int sum = 0;
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // group j = elements 8j .. 8j+7 = words 2j, 2j+1
                o[2 * j] = __byte_perm(w[2 * j], w[2 * j + 1], 0x6420);      // elements 0,2,4,6
                o[2 * j + 1] = __byte_perm(w[2 * j], w[2 * j + 1], 0x7531);  // elements 1,3,5,7
                sum = __dp4a(static_cast<int>(w[2 * j]), 0x01010101, sum);
                sum = __dp4a(static_cast<int>(w[2 * j + 1]), 0x01010101, sum);
            }
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
            dst[8] = static_cast<uint32_t>(sum);
            sdx[i] = __ldg(dx + static_cast<size_t>(t) * nb + b);
        } else {
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(0u, 0u, 0u, 0u);
            dst[8] = 0u;
            sdx[i] = 0.f;
        }
    }
    __syncthreads();

    // ---- row pairs, round-robin over the grid's warps
    const int npairs = (rows + 1) / 2;
    for (int p = blockIdx.x * kWarps + warp; p < npairs; p += gridDim.x * kWarps) {
        const int r0 = 2 * p;
        const bool two = r0 + 1 < rows;
        float acc[2][MT];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[i][t] = 0.f;
        for (int b = lane; b < nb; b += 32) {
            uint32_t q[2][8];  // q bytes in [0, 15], in the staged code order
            float dw[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const size_t idx = static_cast<size_t>(r0 + (i == 1 && two ? 1 : 0)) * nb + b;
                const uint4 v = __ldg(nib + idx);
                dw[i] = (i == 0 || two) ? __half2float(__ushort_as_half(__ldg(dsc + idx))) : 0.f;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    q[i][2 * j] = w[j] & 0x0F0F0F0Fu;             // elements 8j + 0, 2, 4, 6
                    q[i][2 * j + 1] = (w[j] >> 4) & 0x0F0F0F0Fu;  // elements 8j + 1, 3, 5, 7
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint32_t *xs = sx + (static_cast<size_t>(t) * nb + b) * kXW;
                const uint4 x0 = reinterpret_cast<const uint4 *>(xs)[0];
                const uint4 x1 = reinterpret_cast<const uint4 *>(xs)[1];
                const int xsum = static_cast<int>(xs[8]);
                const float d_x = sdx[static_cast<size_t>(t) * nb + b];
                const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    int dot = -8 * xsum;
#pragma unroll
                    for (int j = 0; j < 8; ++j) dot = __dp4a(static_cast<int>(q[i][j]), static_cast<int>(xw[j]), dot);
                    acc[i][t] = fmaf(dw[i] * d_x, static_cast<float>(dot), acc[i][t]);
                }
            }
        }
        // butterfly: every lane ends with every (row, token) sum
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[i][t] += __shfl_xor_sync(0xffffffffu, acc[i][t], o);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (lane == t && t < M) {
                Y[static_cast<size_t>(t) * rows + r0] = acc[0][t];
                if (two) Y[static_cast<size_t>(t) * rows + r0 + 1] = acc[1][t];
            }
        }
    }
}

template <int MT>
size_t smem_bytes(int nb)
{
    return static_cast<size_t>(MT) * nb * (kXW * 4 + 4);
}

}  // namespace small

// Up to 24 tokens, as passes of at most 8 (each pass streams the weights
// again).  Measured on 21504 x 5376 weights: 31.9 us per pass of 8 tokens
// (63.7 us for 16 as two passes, against about 80 us as one 16-token pass),
// while the tensor-core tiles take 123 us at any M <= 128, so three passes
// (95 us) still win and four (128 us) no longer do.  Each pass's staging
// must fit in shared memory.
constexpr int kMaxPass = 8;
constexpr int kMaxTokens = 24;
static size_t pass_smem(int nb, int m) { return m <= 4 ? small::smem_bytes<4>(nb) : small::smem_bytes<8>(nb); }
bool gemm_small_supported(int K, int M)
{
    if (M < 1 || M > kMaxTokens || K < 32 || K % 32 != 0) return false;
    return pass_smem(K / 32, M < kMaxPass ? M : kMaxPass) <= 200 * 1024;
}

int launch_gemm_small(const void *W, const int8_t *Xq, const float *dx, float *Y, int rows, int K, int M,
                      cudaStream_t s)
{
    if (!gemm_small_supported(K, M)) return GQ_ERR_SHAPE;
    const int nb = K / 32;
    const uint4 *nib = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb);
    const long long npairs = (rows + 1) / 2;
    for (int t0 = 0; t0 < M; t0 += kMaxPass) {
        const int m = M - t0 < kMaxPass ? M - t0 : kMaxPass;
        const int8_t *xq = Xq + static_cast<size_t>(t0) * K;
        const float *d = dx + static_cast<size_t>(t0) * nb;
        float *y = Y + static_cast<size_t>(t0) * rows;
        int rc = GQ_OK;
#define GQ_SMALL_CASE(MT)                                                                                       \
    {                                                                                                           \
        const size_t smem = small::smem_bytes<MT>(nb);                                                         \
        const int grid = persistent_grid(reinterpret_cast<const void *>(small::k_gemm_small<MT>), small::kThreads, \
                                         smem, npairs);                                                        \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                                     \
        rc = status_from(launch_pdl(small::k_gemm_small<MT>, dim3(grid), dim3(small::kThreads), smem, s, nib,    \
                                    dsc, xq, d, y, rows, nb, m));                                               \
    }
        if (m <= 4)
            GQ_SMALL_CASE(4)
        else
            GQ_SMALL_CASE(8)
#undef GQ_SMALL_CASE
        if (rc != GQ_OK) return rc;
    }
    return GQ_OK;
}

}  // namespace gq
