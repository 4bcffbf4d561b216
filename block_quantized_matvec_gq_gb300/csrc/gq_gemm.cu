// gq_gemm.cu -- Q4_0 weights x Q8_0 activations prefill contraction.
//
// "Gemma 4 M4 Max kernel roadmap", K3 "prefill path": batched Q4_0
// matrix-matrix kernels sized for the 5376 embedding and the 21504 FFN.
//   D[t][r][b] = sum_{j<32} Xq[t][32b+j] * (q_w[r][32b+j] - 8)   (int32, exact)
//   Y[t][r]    = sum_b d_w[r][b] * dx[t][b] * D[t][r][b]          (f32)
//
// This file holds the integer-dot CUDA-core version: a 64-token x 64-row
// tile per CTA, one 32-block of K per step staged in shared memory, the
// block dot products in int32 with __dp4a, and the scale epilogue in f32.
#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {

constexpr int kGemmTileT = 64;
constexpr int kGemmTileR = 64;

// Four element-order nibbles (16 bits) -> four int8 bytes q - 8.
__device__ __forceinline__ int nib4_to_s8(uint32_t v)
{
    const uint32_t spread = (v & 0xFu) | ((v & 0xF0u) << 4) | ((v & 0xF00u) << 8) | ((v & 0xF000u) << 12);
    return static_cast<int>(__vsub4(spread, 0x08080808u));
}

__global__ void __launch_bounds__(256)
    k_gemm_q8act_dp4a(const uint32_t *__restrict__ nib, const uint16_t *__restrict__ dsc,
                      const int8_t *__restrict__ Xq, const float *__restrict__ dx, float *__restrict__ Y,
                      int rows, int K, int M)
{
    __shared__ int sx[kGemmTileT][9];
    __shared__ int sw[kGemmTileR][9];
    __shared__ float sdx[kGemmTileT], sdw[kGemmTileR];
    const int nb = K / 32;
    const int t0 = blockIdx.y * kGemmTileT, r0 = blockIdx.x * kGemmTileR;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    pdl_wait();
    for (int b = 0; b < nb; ++b) {
        for (int e = tid; e < kGemmTileT * 8; e += 256) {
            const int tt = e >> 3, w = e & 7, t = t0 + tt;
            sx[tt][w] = (t < M) ? reinterpret_cast<const int *>(Xq + static_cast<size_t>(t) * K + b * 32)[w] : 0;
        }
        {
            const int rr = tid >> 2, wq = tid & 3, r = r0 + rr;
            const uint32_t v = (r < rows) ? nib[(static_cast<size_t>(r) * nb + b) * 4 + wq] : 0x88888888u;
            sw[rr][2 * wq] = nib4_to_s8(v & 0xFFFFu);
            sw[rr][2 * wq + 1] = nib4_to_s8(v >> 16);
        }
        if (tid < kGemmTileT) {
            const int t = t0 + tid;
            sdx[tid] = (t < M) ? dx[static_cast<size_t>(t) * nb + b] : 0.f;
        } else if (tid < kGemmTileT + kGemmTileR) {
            const int r = r0 + tid - kGemmTileT;
            sdw[tid - kGemmTileT] = (r < rows) ? __half2float(__ushort_as_half(dsc[static_cast<size_t>(r) * nb + b])) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tt = ty + 16 * i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int rr = tx + 16 * j;
                int dot = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) dot = __dp4a(sx[tt][w], sw[rr][w], dot);
                acc[i][j] = fmaf(sdw[rr] * sdx[tt], static_cast<float>(dot), acc[i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty + 16 * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = r0 + tx + 16 * j;
            if (t < M && r < rows) Y[static_cast<size_t>(t) * rows + r] = acc[i][j];
        }
    }
    pdl_launch_dependents();
}

int launch_gemm_q8act(const void *W, const int8_t *Xq, const float *dx, float *Y, int rows, int K, int M,
                      cudaStream_t s)
{
    const int nb = K / 32;
    const uint32_t *nib = static_cast<const uint32_t *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(
        static_cast<const uint8_t *>(W) + static_cast<size_t>(rows) * nb * 16);
    dim3 grid((rows + kGemmTileR - 1) / kGemmTileR, (M + kGemmTileT - 1) / kGemmTileT);
    return status_from(launch_pdl(k_gemm_q8act_dp4a, grid, dim3(256), 0, s, nib, dsc, Xq, dx, Y, rows, K, M));
}

}  // namespace gq
