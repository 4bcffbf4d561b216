// gq_gemm_tc.cu -- Q4_0 weights x Q8_0 activations on the 5th-generation
// tensor cores (tcgen05), with exact integer block dot products.
//
// "Gemma 4 M4 Max kernel roadmap", K3 "prefill path": batched Q4_0
// matrix-matrix kernels sized for the 5376 embedding and 21504 FFN (there a
// 64-output x 32-prompt SIMD-matrix tile with threadgroup staging).
//   D[t][r][b] = sum_{j<32} Xq[t][32b+j] * (q_w[r][32b+j] - 8)
//   Y[t][r]    = sum_b d_w[r][b] * dx[t][b] * D[t][r][b]
//
// On sm_103a the int8 form of tcgen05.mma is not available, so both
// operands are fed as f16: q_w - 8 in [-8, 7] and Xq in [-127, 127] are
// exact in f16, and every partial sum of a 32-term block dot is an integer
// of magnitude <= 32 * 8 * 127 = 32512 < 2^24, so the f32 accumulator in
// tensor memory holds D exactly.  Because the scales change every 32
// elements, each block's D is read out of tensor memory and folded into the
// f32 result (Y += dx * d_w * D) while the tensor core already computes the
// next block into the other D buffer.
//
// CTA: 576 threads, one per SM, persistent over 128-token x 128-row tiles,
// four 128-column accumulator buffers in TMEM (the MMA runs up to three
// blocks ahead of the epilogue).
//   warps 0-15  workers.  For block g: wait for its D, tcgen05.ld it (warp w
//               owns TMEM lanes 32*(w%4).. and 32 of the 128 columns), fold it
//               into the f32 accumulators, release the D buffer; then convert
//               block g+S from the raw TMA tiles into the f16 UMMA operand
//               layout (the stage the MMA of block g has just finished with)
//               and stage its scales.
//   warp 16     one lane issues the TMA tile loads (int8 codes 128 x 32 B,
//               nibbles 128 x 16 B per block) into an RAW-deep ring.
//   warp 17     one lane issues 2 x (M128 N128 K16) MMAs per block; the warp
//               owns the TMEM allocation.
// Every mbarrier wait is bounded: on timeout the kernel records
// GQ_ERR_TIMEOUT in the device status word, every role leaves its loop, TMEM
// is released and the kernel returns.
#include <cuda.h>

#include "gq_host.h"
#include "gq_internal.cuh"

namespace gq {
namespace tc {

constexpr int TM = 128;  // tokens per tile (MMA M, TMEM lanes)
constexpr int TN = 128;  // weight rows per tile (MMA N, TMEM columns)
constexpr int KB = 32;   // K per quantization block
constexpr int S = 4;     // f16 operand stages
constexpr int SR = 2 * S;  // scale stages
constexpr int RAW = 16;  // raw TMA stages (12 blocks of lead over the conversion)
constexpr int WORK_WARPS = 16;
constexpr int NWORK = WORK_WARPS * 32;
constexpr int TMA_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int NTHREADS = 18 * 32;
constexpr int EPI_COLS = TN / (WORK_WARPS / 4);  // 32
constexpr int NDBUF = 4;     // TMEM accumulator buffers (4 x 128 columns)
constexpr int TMEM_COLS = 512;
constexpr int DBUF = 128;  // TMEM column offset between D buffers

constexpr int A_BYTES = TM * KB * 2;  // 8192: f16 operand A
constexpr int B_BYTES = TN * KB * 2;  // 12288: f16 operand B
constexpr int RA_BYTES = TM * KB;     // 4096: int8 codes (TMA box 32 x 128)
constexpr int RB_BYTES = TN * 16;     // 2048: nibbles (TMA box 16 x 128)
constexpr int RAW_BYTES = RA_BYTES + RB_BYTES;
constexpr int SCL_BYTES = (TM + TN) * 4;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + S * A_BYTES;
constexpr int OFF_RAW = OFF_B + S * B_BYTES;
constexpr int OFF_SCL = OFF_RAW + RAW * RAW_BYTES;
constexpr int OFF_BAR = OFF_SCL + SR * SCL_BYTES;
constexpr int N_BARS = 2 * RAW + S + 2 * NDBUF + 1;  // raw_full, raw_empty, full, dfull, dempty, drain
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16;

static_assert(OFF_B % 1024 == 0 && OFF_RAW % 1024 == 0 && RAW_BYTES % 1024 == 0 && OFF_SCL % 16 == 0 &&
                  OFF_BAR % 8 == 0,
              "alignment");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// A waiting thread may be suspended up to this long inside one try_wait
// (it resumes as soon as the phase completes), so waiting warps do not
// compete with working warps for issue slots.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// Bounded wait for the phase of `bar` with the given parity.  Returns false
// (raising the CTA abort flag and the device status) on timeout, or when
// another role has already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort, int *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicExch(status, GQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// Warp-uniform form (all lanes agree).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort, int *status)
{
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort, status));
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// tcgen05 shared-memory matrix descriptor, K-major, no swizzle: start
// address, LBO = byte stride between core matrices along K, SBO = byte
// stride between 8-row groups along M/N, descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), both K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(TN >> 3) << 17) | (static_cast<uint32_t>(TM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- operand conversion
// Both operands of a 32-block are written as four 8-element K groups; inside
// a group the elements are stored in the order 0,4,1,5,2,6,3,7 (the order in
// which the nibble unpacking below produces them).  A and B use the same
// order, so the dot products are unchanged.
__device__ __forceinline__ uint4 nib8_to_f16(uint32_t w)
{
    const uint32_t w2 = w >> 8;
    uint32_t a0 = (w & 0x000F000Fu) | 0x64006400u;   // 1024 + (e0, e4)
    uint32_t a1 = (w & 0x00F000F0u) | 0x64006400u;   // 1024 + 16 (e1, e5)
    uint32_t a2 = (w2 & 0x000F000Fu) | 0x64006400u;  // 1024 + (e2, e6)
    uint32_t a3 = (w2 & 0x00F000F0u) | 0x64006400u;  // 1024 + 16 (e3, e7)
    const __half2 c1032 = __float2half2_rn(1032.0f);
    const __half2 c16 = __float2half2_rn(0.0625f);
    const __half2 c72 = __float2half2_rn(-72.0f);
    __half2 r0 = __hsub2(*reinterpret_cast<__half2 *>(&a0), c1032);
    __half2 r1 = __hfma2(*reinterpret_cast<__half2 *>(&a1), c16, c72);
    __half2 r2 = __hsub2(*reinterpret_cast<__half2 *>(&a2), c1032);
    __half2 r3 = __hfma2(*reinterpret_cast<__half2 *>(&a3), c16, c72);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t *>(&r0);
    o.y = *reinterpret_cast<uint32_t *>(&r1);
    o.z = *reinterpret_cast<uint32_t *>(&r2);
    o.w = *reinterpret_cast<uint32_t *>(&r3);
    return o;
}
// Eight int8 codes (two words, elements 0..3 and 4..7) -> f16 in group order.
__device__ __forceinline__ uint4 s8x8_to_f16(uint32_t lo, uint32_t hi)
{
    lo ^= 0x80808080u;  // offset binary: u = q + 128
    hi ^= 0x80808080u;
    const uint32_t t01 = __byte_perm(lo, hi, 0x5140);  // u0 u4 u1 u5
    const uint32_t t23 = __byte_perm(lo, hi, 0x7362);  // u2 u6 u3 u7
    uint32_t a0 = __byte_perm(t01, 0x64646464u, 0x4140);  // 1024 + (u0, u4)
    uint32_t a1 = __byte_perm(t01, 0x64646464u, 0x4342);  // 1024 + (u1, u5)
    uint32_t a2 = __byte_perm(t23, 0x64646464u, 0x4140);
    uint32_t a3 = __byte_perm(t23, 0x64646464u, 0x4342);
    const __half2 c = __float2half2_rn(1152.0f);
    __half2 r0 = __hsub2(*reinterpret_cast<__half2 *>(&a0), c);
    __half2 r1 = __hsub2(*reinterpret_cast<__half2 *>(&a1), c);
    __half2 r2 = __hsub2(*reinterpret_cast<__half2 *>(&a2), c);
    __half2 r3 = __hsub2(*reinterpret_cast<__half2 *>(&a3), c);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t *>(&r0);
    o.y = *reinterpret_cast<uint32_t *>(&r1);
    o.z = *reinterpret_cast<uint32_t *>(&r2);
    o.w = *reinterpret_cast<uint32_t *>(&r3);
    return o;
}
// Byte offset of (row, K group kg) in an operand stage: core matrix
// (row/8, kg) at ((row/8)*4 + kg)*128, row%8 at 16-byte steps inside it.
__device__ __forceinline__ uint32_t op_off(int row, int kg) { return (((row >> 3) * 4 + kg) << 7) + ((row & 7) << 4); }

struct Work {
    int ntm, ntiles, nb;
};

// Block gb (running index over this CTA's tiles and their K blocks) -> tile, b.
__device__ __forceinline__ void block_coords(const Work &w, long long gb, int &tile, int &b)
{
    const long long it = gb / w.nb;
    b = static_cast<int>(gb - it * w.nb);
    tile = static_cast<int>(blockIdx.x + it * static_cast<long long>(gridDim.x));
}

// Scales of block gb for this worker thread: thread i < TM loads dx of token i,
// TM <= i < TM + TN loads d_w of row i - TM (0 for rows/tokens past the end).
__device__ __forceinline__ float load_scale(const Work &w, long long gb, int i, const uint16_t *dsc, const float *dx,
                                            int rows, int M)
{
    int tile, b;
    block_coords(w, gb, tile, b);
    const int t0 = (tile % w.ntm) * TM, r0 = (tile / w.ntm) * TN;
    if (i < TM) {
        const int t = t0 + i;
        return (t < M && dx != nullptr) ? __ldg(dx + static_cast<size_t>(t) * w.nb + b) : 0.f;
    }
    if (i < TM + TN) {
        const int r = r0 + i - TM;
        return (r < rows) ? __half2float(__ushort_as_half(__ldg(dsc + static_cast<size_t>(r) * w.nb + b))) : 0.f;
    }
    return 0.f;
}

// Convert raw block (codes, nibbles) into the f16 operand stage.
__device__ __forceinline__ void convert_block(const uint8_t *raw, uint8_t *opA, uint8_t *opB, int tid)
{
#pragma unroll
    for (int k = 0; k < (TM * 4 + TN * 4 + NWORK - 1) / NWORK; ++k) {
        const int i = tid + k * NWORK;
        if (i < TM * 4) {
            const int row = i % TM, kg = i / TM;
            const uint2 v = *reinterpret_cast<const uint2 *>(raw + row * 32 + kg * 8);
            *reinterpret_cast<uint4 *>(opA + op_off(row, kg)) = s8x8_to_f16(v.x, v.y);
        } else if (i < TM * 4 + TN * 4) {
            const int j = i - TM * 4;
            const int row = j % TN, kg = j / TN;
            const uint32_t v = *reinterpret_cast<const uint32_t *>(raw + RA_BYTES + row * 16 + kg * 4);
            *reinterpret_cast<uint4 *>(opB + op_off(row, kg)) = nib8_to_f16(v);
        }
    }
}

// ---------------------------------------------------------------- the kernel
template <bool kDumpD>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_q8act_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const uint16_t *__restrict__ dsc, const float *__restrict__ dx, float *__restrict__ Y,
                    int32_t *__restrict__ Dout, int rows, int K, int M, int *__restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_rfull = sbase + OFF_BAR, bar_rempty = bar_rfull + 8 * RAW;
    const uint32_t bar_full = bar_rempty + 8 * RAW, bar_dfull = bar_full + 8 * S;
    const uint32_t bar_dempty = bar_dfull + 8 * NDBUF, bar_drain = bar_dempty + 8 * NDBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    Work w;
    w.nb = K / KB;
    w.ntm = (M + TM - 1) / TM;
    w.ntiles = w.ntm * ((rows + TN - 1) / TN);
    const int my_tiles = (w.ntiles > static_cast<int>(blockIdx.x))
                             ? (w.ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const long long nblocks = static_cast<long long>(my_tiles) * w.nb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RAW; ++i) {
            mbar_init(bar_rfull + 8 * i, 1);
            mbar_init(bar_rempty + 8 * i, WORK_WARPS);
        }
        for (int s = 0; s < S; ++s) mbar_init(bar_full + 8 * s, WORK_WARPS);
        for (int b = 0; b < NDBUF; ++b) {
            mbar_init(bar_dfull + 8 * b, 1);
            mbar_init(bar_dempty + 8 * b, WORK_WARPS);
        }
        mbar_init(bar_drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    if (warp == TMA_WARP) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (long long gb = 0; gb < nblocks; ++gb) {
                const int rs = static_cast<int>(gb % RAW);
                if (!wait_bounded(bar_rempty + 8 * rs, static_cast<uint32_t>(((gb / RAW) & 1) ^ 1), abort, status))
                    break;
                int tile, b;
                block_coords(w, gb, tile, b);
                const int t0 = (tile % w.ntm) * TM, r0 = (tile / w.ntm) * TN;
                const uint32_t raw = sbase + OFF_RAW + rs * RAW_BYTES;
                mbar_expect_tx(bar_rfull + 8 * rs, RAW_BYTES);
                tma_load_2d(raw, &mapA, b * KB, t0, bar_rfull + 8 * rs);
                tma_load_2d(raw + RA_BYTES, &mapB, b * 16, r0, bar_rfull + 8 * rs);
            }
            // No tile load may still be landing in shared memory when the CTA exits
            // (relevant only after an abort: normally every load has been consumed).
            volatile int no_abort = 0;
            for (long long gb = (nblocks > RAW ? nblocks - RAW : 0); gb < nblocks; ++gb)
                wait_bounded(bar_rfull + 8 * static_cast<int>(gb % RAW), static_cast<uint32_t>((gb / RAW) & 1),
                             &no_abort, status);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (long long gb = 0; gb < nblocks; ++gb) {
                const int s = static_cast<int>(gb % S);
                const int buf = static_cast<int>(gb % NDBUF);
                if (!wait_bounded(bar_full + 8 * s, static_cast<uint32_t>((gb / S) & 1), abort, status)) break;
                if (!wait_bounded(bar_dempty + 8 * buf, static_cast<uint32_t>(((gb / NDBUF) & 1) ^ 1), abort, status))
                    break;
                tc_fence_after();
                const uint32_t a0 = sbase + OFF_A + s * A_BYTES, b0 = sbase + OFF_B + s * B_BYTES;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_f16(tmem + buf * DBUF, smem_desc(a0 + ks * 256, 128, 512), smem_desc(b0 + ks * 256, 128, 512),
                            ks);
                mma_commit(bar_dfull + 8 * buf);
            }
            // every issued MMA has completed before tensor memory is released
            mma_commit(bar_drain);
            wait_bounded(bar_drain, 0u, abort, status);
        }
        __syncwarp();
    } else if (warp < WORK_WARPS) {
        // ------------------------------------------------ workers
        const int tid = threadIdx.x;  // 0..NWORK-1
        const int q = warp & 3;       // TMEM lane quarter
        const int c0 = (warp >> 2) * EPI_COLS;
        bool ok = true;
        // stage blocks 0..S-1
        for (long long gb = 0; gb < S && gb < nblocks && ok; ++gb) {
            const int rs = static_cast<int>(gb % RAW);
            const float sv = load_scale(w, gb, tid, dsc, dx, rows, M);
            ok = wait_warp(bar_rfull + 8 * rs, static_cast<uint32_t>((gb / RAW) & 1), abort, status);
            if (!ok) break;
            convert_block(smem + OFF_RAW + rs * RAW_BYTES, smem + OFF_A + (gb % S) * A_BYTES,
                          smem + OFF_B + (gb % S) * B_BYTES, tid);
            if (tid < TM + TN) reinterpret_cast<float *>(smem + OFF_SCL + (gb % SR) * SCL_BYTES)[tid] = sv;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_full + 8 * (gb % S));
                mbar_arrive(bar_rempty + 8 * rs);
            }
        }
        float acc[EPI_COLS];
#pragma unroll
        for (int c = 0; c < EPI_COLS; ++c) acc[c] = 0.f;
        // scales are loaded one iteration before they are staged
        float sv_next = (S < nblocks) ? load_scale(w, S, tid, dsc, dx, rows, M) : 0.f;
        for (long long gb = 0; gb < nblocks && ok; ++gb) {
            const int buf = static_cast<int>(gb % NDBUF);
            const long long gn = gb + S;  // block converted in this iteration
            const float sv = sv_next;
            sv_next = (gn + 1 < nblocks) ? load_scale(w, gn + 1, tid, dsc, dx, rows, M) : 0.f;
            ok = wait_warp(bar_dfull + 8 * buf, static_cast<uint32_t>((gb / NDBUF) & 1), abort, status);
            if (!ok) break;
            tc_fence_after();
            int tile, b;
            block_coords(w, gb, tile, b);
            const int t0 = (tile % w.ntm) * TM, r0 = (tile / w.ntm) * TN;
            const float *scl = reinterpret_cast<const float *>(smem + OFF_SCL + (gb % SR) * SCL_BYTES);
            const float dxt = scl[q * 32 + lane];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * DBUF + c0;
#pragma unroll
            for (int part = 0; part < EPI_COLS / 16; ++part) {
                float d[16];
                tmem_ld16(taddr + part * 16, d);
                if (part == EPI_COLS / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_dempty + 8 * buf);
                }
                if (kDumpD) {
                    const int t = t0 + q * 32 + lane;
                    if (t < M) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int r = r0 + c0 + part * 16 + c;
                            if (r < rows) Dout[(static_cast<size_t>(t) * rows + r) * w.nb + b] = __float2int_rz(d[c]);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; c += 4) {
                        const int cc = part * 16 + c;
                        const float4 wv = *reinterpret_cast<const float4 *>(scl + TM + c0 + cc);
                        const float2 s01 = __fmul2_rn(make_float2(dxt, dxt), make_float2(wv.x, wv.y));
                        const float2 s23 = __fmul2_rn(make_float2(dxt, dxt), make_float2(wv.z, wv.w));
                        float2 a01 = __ffma2_rn(s01, make_float2(d[c], d[c + 1]), make_float2(acc[cc], acc[cc + 1]));
                        float2 a23 = __ffma2_rn(s23, make_float2(d[c + 2], d[c + 3]), make_float2(acc[cc + 2], acc[cc + 3]));
                        acc[cc] = a01.x;
                        acc[cc + 1] = a01.y;
                        acc[cc + 2] = a23.x;
                        acc[cc + 3] = a23.y;
                    }
                }
            }
            if (!kDumpD && b == w.nb - 1) {
                const int t = t0 + q * 32 + lane;
                if (t < M) {
                    float *yrow = Y + static_cast<size_t>(t) * rows + r0 + c0;
                    const int nvalid = rows - (r0 + c0);
                    if (nvalid >= EPI_COLS && (rows & 3) == 0) {
#pragma unroll
                        for (int c = 0; c < EPI_COLS; c += 4)
                            *reinterpret_cast<float4 *>(yrow + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                    } else {
#pragma unroll
                        for (int c = 0; c < EPI_COLS; ++c)
                            if (c < nvalid) yrow[c] = acc[c];
                    }
                }
#pragma unroll
                for (int c = 0; c < EPI_COLS; ++c) acc[c] = 0.f;
            }
            // convert block gb + S into the stage the MMA of block gb has finished with
            if (gn < nblocks) {
                const int rs = static_cast<int>(gn % RAW);
                ok = wait_warp(bar_rfull + 8 * rs, static_cast<uint32_t>((gn / RAW) & 1), abort, status);
                if (!ok) break;
                convert_block(smem + OFF_RAW + rs * RAW_BYTES, smem + OFF_A + (gn % S) * A_BYTES,
                              smem + OFF_B + (gn % S) * B_BYTES, tid);
                if (tid < TM + TN) reinterpret_cast<float *>(smem + OFF_SCL + (gn % SR) * SCL_BYTES)[tid] = sv;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_full + 8 * (gn % S));
                    mbar_arrive(bar_rempty + 8 * rs);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace tc

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor [outer][inner] with row stride `stride` bytes; box inner x outer.
static bool make_map_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t stride,
                        uint32_t box_inner, uint32_t box_outer)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int launch_tc(bool dump, const void *W, const int8_t *Xq, const float *dx, float *Y, int32_t *D, int rows,
                     int K, int M, cudaStream_t s)
{
    const int nb = K / 32;
    const uint8_t *nib = static_cast<const uint8_t *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb * 16);
    CUtensorMap mapA, mapB;
    if (!make_map_u8(&mapA, Xq, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K), tc::KB,
                     tc::TM))
        return GQ_ERR_CUDA;
    if (!make_map_u8(&mapB, nib, static_cast<uint64_t>(nb) * 16, static_cast<uint64_t>(rows),
                     static_cast<uint64_t>(nb) * 16, 16, tc::TN))
        return GQ_ERR_CUDA;
    const int ntiles = ((M + tc::TM - 1) / tc::TM) * ((rows + tc::TN - 1) / tc::TN);
    auto kern = dump ? tc::k_gemm_q8act_tc<true> : tc::k_gemm_q8act_tc<false>;
    const int occ = ctas_per_sm(reinterpret_cast<const void *>(kern), tc::NTHREADS, tc::SMEM_BYTES);
    if (occ <= 0) return GQ_ERR_CUDA;
    int grid = sm_count();
    if (grid > ntiles) grid = ntiles;
    return status_from(launch_pdl(kern, dim3(grid), dim3(tc::NTHREADS), static_cast<size_t>(tc::SMEM_BYTES), s, mapA,
                                  mapB, dsc, dx, Y, D, rows, K, M, status_word()));
}

int launch_gemm_q8act_tc(const void *W, const int8_t *Xq, const float *dx, float *Y, int rows, int K, int M,
                         cudaStream_t s)
{
    return launch_tc(false, W, Xq, dx, Y, nullptr, rows, K, M, s);
}

int launch_block_dots_tc(const void *W, const int8_t *Xq, int32_t *D, int rows, int K, int M, cudaStream_t s)
{
    return launch_tc(true, W, Xq, nullptr, nullptr, D, rows, K, M, s);
}

}  // namespace gq
