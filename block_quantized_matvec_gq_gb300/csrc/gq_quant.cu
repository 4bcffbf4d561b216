// gq_quant.cu -- Q8_0 quantization of f32 activations (one warp per 32-block).
//
// "Metal kernel capability table (Phase B ground truth)", section 2
// (quantize_q8: f32 -> int8 plus per-32 external scales) and finding F6
// (every block's scale must be written; here K % 32 == 0 is required and
// each 32-block is one warp, so no tail scale can be left unwritten).
//   amax = max |x|, d = amax / 127, q = clamp(round_half_away(x / d), -127, 127)
// with IEEE-rounded f32 division; d = 0 gives q = 0.
#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {

__global__ void __launch_bounds__(256)
    k_quantize_q8_0(const float *__restrict__ X, int8_t *__restrict__ Xq, float *__restrict__ dx,
                    long long nblocks)
{
    const int lane = threadIdx.x & 31;
    // dependents launch once every CTA of this grid has started; they still
    // wait for its completion before reading Xq and dx
    pdl_launch_dependents();
    pdl_wait();
    for (long long blk = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; blk < nblocks;
         blk += ((long long)gridDim.x * blockDim.x) >> 5) {
        const float v = X[blk * 32 + lane];
        float amax = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        int q = 0;
        if (d != 0.0f) {
            float r = roundf(__fdiv_rn(v, d));
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q = static_cast<int>(r);
        }
        Xq[blk * 32 + lane] = static_cast<int8_t>(q);
        if (lane == 0) dx[blk] = d;
    }
}

int launch_quantize_q8_0(const float *X, int8_t *Xq, float *dx, int K, int M, cudaStream_t s)
{
    // The [M][K] row-major X is a sequence of M*K/32 consecutive 32-blocks,
    // and dx[M][K/32] lists their scales in the same order.
    const long long nblocks = (long long)M * (K / 32);
    const int threads = 256;
    long long grid = (nblocks * 32 + threads - 1) / threads;
    const long long cap = (long long)sm_count() * 8;
    if (grid > cap) grid = cap;
    return status_from(launch_pdl(k_quantize_q8_0, dim3((unsigned)grid), dim3(threads), 0, s, X, Xq,
                                  dx, nblocks));
}

}  // namespace gq
