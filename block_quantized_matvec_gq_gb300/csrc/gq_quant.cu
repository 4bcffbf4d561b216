// gq_quant.cu -- Q8_0 quantization of f32 activations (eight lanes per 32-block).
//
// "Metal kernel capability table (Phase B ground truth)", section 2
// (quantize_q8: f32 -> int8 plus per-32 external scales) and finding F6
// (every block's scale must be written; here K % 32 == 0 is required and
// each 32-block is one group of eight lanes, so no tail scale can be left
// unwritten).
//   amax = max |x|, d = amax / 127, q = clamp(round_half_away(x / d), -127, 127)
// with IEEE-rounded f32 division; d = 0 gives q = 0.
#include "gq_host.h"
#include "gq_internal.cuh"
#include "gq_q8code.cuh"

namespace gq {

// Eight lanes per 32-block, four consecutive elements per lane (16-byte
// loads, 4-byte code stores); the codes follow q8_pack4 (one reciprocal per
// block, full-rate arithmetic, the division itself next to a half-integer).
__global__ void __launch_bounds__(256)
    k_quantize_q8_0(const float4 *__restrict__ X, uint32_t *__restrict__ Xq, float *__restrict__ dx,
                    long long nblocks)
{
    const int sub = threadIdx.x & 7;  // which four elements of the block this lane holds
    // dependents launch once every CTA of this grid has started; they still
    // wait for its completion before reading Xq and dx
    pdl_launch_dependents();
    pdl_wait();
    // warp-uniform loop over groups of four blocks (the shuffles below use the
    // full warp), a block per eight lanes
    for (long long wb = ((blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5) * 4; wb < nblocks;
         wb += ((long long)gridDim.x * blockDim.x) >> 3) {
        const long long blk = wb + ((threadIdx.x & 31) >> 3);
        const bool active = blk < nblocks;
        const float4 v = active ? __ldg(X + blk * 8 + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
        float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float d = __fdiv_rn(amax, 127.0f);
        const float e[4] = {v.x, v.y, v.z, v.w};
        const uint32_t packed = q8_pack4(e, d);
        if (active) {
            Xq[blk * 8 + sub] = packed;
            if (sub == 0) dx[blk] = d;
        }
    }
}

int launch_quantize_q8_0(const float *X, int8_t *Xq, float *dx, int K, int M, cudaStream_t s)
{
    // The [M][K] row-major X is a sequence of M*K/32 consecutive 32-blocks,
    // and dx[M][K/32] lists their scales in the same order.  X and Xq are
    // 16-byte aligned (checked by the caller).
    const long long nblocks = (long long)M * (K / 32);
    const int threads = 256;
    long long grid = (nblocks * 8 + threads - 1) / threads;
    const long long cap = (long long)sm_count() * 16;
    if (grid > cap) grid = cap;
    return status_from(launch_pdl(k_quantize_q8_0, dim3((unsigned)grid), dim3(threads), 0, s,
                                  reinterpret_cast<const float4 *>(X), reinterpret_cast<uint32_t *>(Xq), dx,
                                  nblocks));
}

}  // namespace gq
