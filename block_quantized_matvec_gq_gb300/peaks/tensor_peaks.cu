// tensor_peaks.cu -- measured peaks of the tensor paths the contraction can
// use on this GPU (sm_103a), for the roofline denominators:
//   * tcgen05.mma kind::f16 (f16 x f16 -> f32 in tensor memory), M=128 N=256
//     K=16 per instruction, one issuing thread per CTA, one CTA per SM;
//   * tcgen05.ld read-out rate (tensor memory -> registers, 32x32b.x64), the
//     rate that bounds a contraction which reads its accumulators out often;
//   * mma.sync m16n8k16 f16 -> f32 and m16n8k32 s8 -> s32 (the register-
//     operand tensor path), 16 warps per SM, eight independent accumulators;
//   * f32 FMA rate on the CUDA cores, scalar and packed (fma.rn.f32x2): the
//     rate that bounds a per-block scale epilogue (two f32 operations per
//     accumulator element and block).
// Operands are whatever shared memory and registers hold: only the rates
// are measured.  Every wait is bounded (a timeout sets a flag and the probe
// reports it instead of a number).  Prints one JSON object.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "gq_tc.cuh"

using namespace gq;
using namespace gq::tcu;

namespace {

constexpr int kCols = 256;  // N = 256 f32 accumulator columns

__device__ int g_timeout;

// One CTA per SM, 512 threads; thread 0 issues `iters` MMAs (accumulating
// into the same 128 x 256 tile), commits them to an mbarrier; all wait.
// Then the sixteen warps read the tile out of tensor memory `reads` times
// (warp w: TMEM lanes 32 (w % 4).., columns 64 (w / 4)..; one x64 load per
// warp and read, so sixteen loads are in flight per SM).
__global__ void __launch_bounds__(512, 1) k_umma(int iters, int reads, float *sink)
{
    __shared__ __align__(1024) uint8_t opA[128 * 64];  // 128 rows x 32 K f16
    __shared__ __align__(1024) uint8_t opB[256 * 64];  // 256 rows x 32 K f16
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 128 * 64 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(opA)[i] = 0x3C003C00u;
    for (int i = threadIdx.x; i < 256 * 64 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(opB)[i] = 0x3C003C00u;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_async_smem();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // K-major, no swizzle: core matrices of 8 rows x 16 B; four K groups per
    // 8-row group (LBO 128 B along K, SBO 512 B along M/N)
    const uint32_t a0 = smem_u32(opA), b0 = smem_u32(opB);
    const uint32_t idesc = idesc_f16(128, 256, false);
    if (threadIdx.x == 0) {
        for (int i = 0; i < iters; ++i) {
            const uint32_t koff = (i & 1) ? 256u : 0u;  // K half of the stored 32
            mma_f16(tmem, smem_desc(a0 + koff, 128, 512), smem_desc(b0 + koff, 128, 512), idesc, i > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar));
    }
    __syncwarp();
    // bounded wait for the MMAs
    {
        const uint64_t t0 = globaltimer();
        bool ok = false;
        while (!ok) {
            ok = mbar_try_wait(smem_u32(&bar), 0);
            if (!ok && globaltimer() - t0 > 2000000000ull) {
                atomicExch(&g_timeout, 1);
                break;
            }
        }
    }
    tc_fence_after();
    float acc = 0.f;
    for (int r = 0; r < reads; ++r) {
        uint32_t v[64];
        const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + static_cast<uint32_t>((warp >> 2) * 64);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
            "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
              "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
              "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
              "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
              "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
              "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 64; ++j) acc += __uint_as_float(v[j]);
    }
    sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
}

// mma.sync: 16 warps per CTA, eight independent accumulator tiles per warp.
template <bool kS8>
__global__ void __launch_bounds__(512, 1) k_mma_sync(int iters, float *sink)
{
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * (threadIdx.x & 3) + i;
    b[0] = 0x00010001u * (threadIdx.x & 7);
    b[1] = b[0] + 3;
    uint32_t d[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) d[t][j] = 0u;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (kS8)
                asm volatile(
                    "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(d[t][0]), "+r"(d[t][1]), "+r"(d[t][2]), "+r"(d[t][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
            else
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(d[t][0]), "+r"(d[t][1]), "+r"(d[t][2]), "+r"(d[t][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
    }
    uint32_t s = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) s ^= d[t][j];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = __uint_as_float(s);
}

// f32 FMA rate: 16 warps per CTA, eight independent chains per thread.
template <bool kPacked>
__global__ void __launch_bounds__(512, 1) k_ffma(int iters, float *sink)
{
    float a[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = 1.0f + 1e-3f * (threadIdx.x + j);
    const float m = 0.999f, c = 1e-6f;
    for (int it = 0; it < iters; ++it) {
        if (kPacked) {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                float2 v = make_float2(a[j], a[j + 1]);
                v = __ffma2_rn(v, make_float2(m, m), make_float2(c, c));
                a[j] = v.x;
                a[j + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = fmaf(a[j], m, c);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += a[j];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <typename F>
float time_ms(F launch)
{
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    launch();  // warm
    cudaEventRecord(e0);
    launch();
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return ms;
}

}  // namespace

int main()
{
    int sms = 0, clk_khz = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
    float *sink = nullptr;
    if (cudaMalloc(&sink, static_cast<size_t>(sms) * 512 * sizeof(float)) != cudaSuccess) return 1;  // 512 threads
    const int zero = 0;
    cudaMemcpyToSymbol(g_timeout, &zero, sizeof zero);

    // tcgen05 kind::f16: 128 x 256 x 16 per instruction
    const int iters = 20000;
    const float ms_mma = time_ms([&] { k_umma<<<sms, 512>>>(iters, 0, sink); });
    const double flops_mma = 2.0 * 128 * 256 * 16 * static_cast<double>(iters) * sms;
    // tcgen05.ld read-out: the same launch with few MMAs and many reads
    const int reads = 2000;
    const float ms_rd = time_ms([&] { k_umma<<<sms, 512>>>(1, reads, sink); });
    const double bytes_rd = 128.0 * kCols * 4 * reads * sms;  // each read: the whole 128 x 256 tile
    // mma.sync
    const int it2 = 20000;
    const float ms_f16 = time_ms([&] { k_mma_sync<false><<<sms, 512>>>(it2, sink); });
    const float ms_s8 = time_ms([&] { k_mma_sync<true><<<sms, 512>>>(it2, sink); });
    const double per_warp_iter = 8.0 * sms * 16 * it2;
    const double flops_f16 = per_warp_iter * 2 * 16 * 8 * 16;
    const double ops_s8 = per_warp_iter * 2 * 16 * 8 * 32;
    const int it3 = 20000;
    const float ms_ffma = time_ms([&] { k_ffma<false><<<sms, 512>>>(it3, sink); });
    const float ms_ffma2 = time_ms([&] { k_ffma<true><<<sms, 512>>>(it3, sink); });
    const double fma_count = 16.0 * 512 * sms * it3;
    const cudaError_t e = cudaDeviceSynchronize();
    int timeout = 0;
    cudaMemcpyFromSymbol(&timeout, g_timeout, sizeof timeout);
    printf("{\"sms\": %d, \"clock_khz_attr\": %d, \"status\": \"%s\", \"timeout\": %d,\n", sms, clk_khz,
           cudaGetErrorString(e), timeout);
    printf(" \"tcgen05_f16_tflops\": %.1f, \"tcgen05_f16_ms\": %.3f,\n", flops_mma / ms_mma / 1e9, ms_mma);
    printf(" \"tcgen05_ld_tb_per_s\": %.2f, \"tcgen05_ld_bytes_per_sm_clk_at_attr\": %.1f,\n",
           bytes_rd / ms_rd / 1e9, bytes_rd / sms / (ms_rd * 1e-3) / (clk_khz * 1e3));
    printf(" \"mma_sync_f16_tflops\": %.1f, \"mma_sync_s8_tops\": %.1f,\n", flops_f16 / ms_f16 / 1e9,
           ops_s8 / ms_s8 / 1e9);
    printf(" \"ffma_scalar_tfma_per_s\": %.2f, \"ffma_packed_tfma_per_s\": %.2f}\n", fma_count / ms_ffma / 1e9,
           fma_count / ms_ffma2 / 1e9);
    return (e == cudaSuccess && timeout == 0) ? 0 : 1;
}
