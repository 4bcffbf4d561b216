// gq_gemm_split.cu -- the prefill contraction with both block scales folded
// into the tensor-core operands, so Y accumulates in tensor memory across
// 8 blocks at a time (one read-out per 8 blocks instead of one per block).
//
// "Gemma 4 M4 Max kernel roadmap", K3 "prefill path" (batched Q4_0
// matrix-matrix):  Y[t][r] = sum_b d_w[r][b] * dx[t][b] * D[t][r][b]
// with D the integer dot of block b.  Over one chunk c of 8 blocks
// (256 values of k) this is one sum over k,
//   Y_c[t][r] = 2^-(s_t + u_r) * sum_k A'[t][k] * B'[r][k],
//   A'[t][k] = (dx[t][k/32] * 2^s_t) * Xq[t][k]       (f32: one rounding, 2^-24)
//   B'[r][k] = (d_w[r][k/32] * 2^u_r) * (q_w[r][k] - 8) (exact: 11 x 3 bits)
// with power-of-two exponents s_t (per token and chunk) and u_r (per row and
// chunk) chosen from the chunk's largest scale so that |A'| < 2^15 and
// |B'| < 2^15 (f16 range, normal numbers down to the chunk's small values).
// The operands are fed to kind::f16 MMAs as f16 pieces: B' = B1 + B2
// exactly (14 significant bits), A' = A1 + A2 to 22 bits.  Three products
// per K step (A1B1, A1B2, A2B1) leave out A2*B2 and the A remainder, both
// below 2^-22 relative; every piece product is exact.  The tensor core's
// f32 accumulation truncates (each add errs toward zero), so each chunk's
// accumulator is read out (24 MMAs per 128 K) and added into f32 registers
// with round-to-nearest, times its power-of-two factor 2^-(s_t + u_r).
// The result equals the block-scaled sum up to f32 rounding, like the
// per-block fold, at three times the tensor work and one eighth of the
// read-outs.
//
// Requires K % 256 == 0 (8-block chunks and scale tiles); other K use the
// per-block fold in gq_gemm_tc.cu.  With more than 128 tokens the CTA-pair
// kernel (k_gemm_pair, one M = 256 MMA per pair of SMs) is used.
//
// Kernels:
//   k_xq_split   writes A1, A2 into the caller's workspace, one 16 KB chunk
//                per (128-token tile, 32-block) in the UMMA K-major layout
//                (f16, 8-element groups in the order 0,4,1,5,2,6,3,7).
//   k_gemm_split one 608-thread CTA per SM, persistent over 128-token x
//                192-row tiles, two 8-block chunk accumulators in TMEM:
//   warps 0-11  read-out: after each 8-block chunk, add its accumulator
//               times 2^-(s_t + u_r) into f32 registers (warp w: TMEM lanes
//               32*(w%4).., 64 of the 192 columns) and store Y after a
//               tile's last chunk.
//   warps 12-15 converters: for each block, build B1, B2 from the nibbles
//               and the d_w scale tile into the operand stage the MMA of
//               block g-S has released (each thread: 3 rows x 16 weights);
//               at a chunk's start, its rows' 2^-u_r for the read-out.
//   warp 16     one lane: TMA loads of the 192 x 16 B nibbles per block
//               and, every 8 blocks, of the 8 x 192 d_w scale tile.
//   warp 17     one lane: 6 MMAs (M128 N192 K16) per block into the
//               chunk's accumulator; owns TMEM.
//   warp 18     one lane: bulk copy of each block's 16 KB A chunk.
// The read-out runs on its own warps, so the conversion (the path's
// limiter: it is latency-bound, one converter warp per scheduler) never
// waits for it.
// Every mbarrier wait is bounded (see gq_tc.cuh): on timeout the kernel
// records GQ_ERR_TIMEOUT, every role leaves its loop, TMEM is released.
#include <cuda_fp16.h>

#include "gq_tc.cuh"

namespace gq {
namespace tcs {

using namespace tcu;

constexpr int TM = 128;   // tokens per tile (MMA M, TMEM lanes)
constexpr int TN = 192;   // weight rows per tile (MMA N, TMEM columns)
constexpr int KB = 32;    // K per quantization block
constexpr int S = 4;      // operand stages
constexpr int RAW = 8;    // raw nibble stages
constexpr int SG = 8;     // blocks per scale tile
constexpr int STG = 2;    // scale tile stages
constexpr int RO_WARPS = 12;    // read-out warps: 4 TMEM lane quarters x 3 column groups
constexpr int CONV_WARPS = 4;   // converter warps (weight pieces)
constexpr int CONV0 = RO_WARPS; // first converter warp
constexpr int TMA_WARP = RO_WARPS + CONV_WARPS;
constexpr int MMA_WARP = TMA_WARP + 1;
constexpr int ACOPY_WARP = TMA_WARP + 2;
constexpr int NTHREADS = (ACOPY_WARP + 1) * 32;  // 608: up to 104 registers per thread
constexpr int EPI_COLS = TN / (RO_WARPS / 4);    // 64
constexpr int CROWS = TN / 64;                   // rows per converter thread (two nibble words each)
constexpr int NACC = 2;          // chunk accumulators (a chunk = SG blocks)
constexpr int ACC_STRIDE = 256;  // TMEM column offset between them
constexpr int TMEM_COLS = 512;

constexpr int APIECE = TM * KB * 2;   // 8192: one f16 piece of A
constexpr int A_BYTES = 2 * APIECE;   // 16384: one workspace chunk
constexpr int BPIECE = TN * KB * 2;   // 12288: one f16 piece of B
constexpr int B_BYTES = 2 * BPIECE;   // 24576
constexpr int RB_BYTES = TN * 16;     // 3072: nibbles (TMA box 16 x 192)
constexpr int STW_BYTES = TN * SG * 2;  // 3072: d_w fp16 [192 rows][8 blocks]
constexpr int NSR = 4;                  // chunks of row factors in flight
constexpr int SR_BYTES = TN * 4;        // 2^-u_r of the tile's 192 rows for one chunk

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + S * A_BYTES;
constexpr int OFF_RAW = OFF_B + S * B_BYTES;
constexpr int OFF_STILE = OFF_RAW + RAW * RB_BYTES;
constexpr int OFF_SR = OFF_STILE + STG * STW_BYTES;
constexpr int OFF_BAR = OFF_SR + NSR * SR_BYTES;
// afull, opempty, full per operand stage; rfull, rempty per raw stage;
// cfull, cempty per chunk accumulator; sfull, sempty per scale tile stage;
// srdy per row-factor slot; drain
constexpr int N_BARS = 3 * S + 2 * RAW + 2 * NACC + 2 * STG + NSR + 1;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16;

static_assert((S & (S - 1)) == 0 && (RAW & (RAW - 1)) == 0 && (SG & (SG - 1)) == 0 && (STG & (STG - 1)) == 0 &&
                  (NACC & (NACC - 1)) == 0 && (NSR & (NSR - 1)) == 0,
              "ring sizes are powers of two");
static_assert(OFF_B % 1024 == 0 && OFF_RAW % 1024 == 0 && OFF_STILE % 128 == 0 && OFF_SR % 16 == 0 &&
                  OFF_BAR % 8 == 0 && SMEM_BYTES <= 232448,
              "shared memory layout");
static_assert(CONV_WARPS == 4 && TN % 64 == 0, "converter warp v: words 2h, 2h+1 (h = v % 2), rows 32 * (v / 2) + 64 * k + lane");

constexpr uint32_t kIdesc = idesc_f16(TM, TN, false);  // f16 A and B
constexpr uint32_t kNegB = 1u << 14;  // instruction descriptor: negate B (the stored second weight piece is -B2)

// ---------------------------------------------------------------- chunk exponents
// Exponents of the power-of-two chunk factors: for m > 0 (the chunk's
// largest scale), m * 2^e lies in [2^(T-1), 2^T); e = 0 for m = 0, NaN or
// infinity.  Read from the IEEE bits (subnormal m counts as 2^-126) and
// clamped to [-60, 60], so 2^e, 2^-e and 2^-(s_t + u_r) are normal floats.
constexpr int kTokExp = 8;    // max |A'| < 127 * 2^8 < 2^15
constexpr int kRowExp = 12;   // max |B'| <= 8 * 2^12 = 2^15
__device__ __forceinline__ int chunk_exp(float m, int T)
{
    const uint32_t bits = __float_as_uint(m);
    const int be = static_cast<int>((bits >> 23) & 0xFFu);
    if (!(m > 0.f) || be == 0xFF) return 0;
    const int e = (be == 0 ? 1 : be) - 126;  // m in [2^(e-1), 2^e)
    const int x = T - e;
    return x < -60 ? -60 : (x > 60 ? 60 : x);
}
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Largest of 8 block scales: dx f32 (non-negative, from amax / 127) or d_w fp16 (|d|).
__device__ __forceinline__ float max8_f32(float4 a, float4 b)
{
    return fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
}
__device__ __forceinline__ float max8_f16(uint4 v)
{
    float m = 0.f;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xFFFFu)))));
        m = fmaxf(m, fabsf(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16)))));
    }
    return m;
}

// ---------------------------------------------------------------- operand pieces
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// (a, b) -> f16x2 hi = RN(a, b) and the exact remainders (a - hi.x, b - hi.y).
__device__ __forceinline__ uint32_t split_h2(float a, float b, float &ra, float &rb)
{
    const __half2 h = __floats2half2_rn(a, b);
    ra = a - __low2float(h);
    rb = b - __high2float(h);
    return h2_bits(h);
}

// Activation pieces: thread p writes 16 bytes of each piece of chunk p/512
// = (token tile T, block b), T-major, at 8-element group position p % 512
// (= op_off(row, kg) / 16).  Tokens past M are zeros.  The thread of group
// 0 of a chunk's first block also writes the token's chunk factor 2^-s_t
// to tokf[token][chunk] (1 for tokens past M).
__global__ void __launch_bounds__(256) k_xq_split(const int8_t *__restrict__ Xq, const float *__restrict__ dx,
                                                  uint4 *__restrict__ Xh, float *__restrict__ tokf, int K, int M,
                                                  long long npieces)
{
    pdl_launch_dependents();  // the GEMM's prologue may overlap; it waits for this grid before reading Xh
    pdl_wait();
    const int nb = K / KB;
    for (long long p = blockIdx.x * 256ll + threadIdx.x; p < npieces; p += static_cast<long long>(gridDim.x) * 256) {
        const long long chunk = p >> 9;
        const int within = static_cast<int>(p & 511);
        const int row = ((within >> 5) << 3) | (within & 7), kg = (within >> 3) & 3;
        const long long T = chunk / nb;
        const int b = static_cast<int>(chunk - T * nb);
        const long long t = T * TM + row;
        uint4 o1 = make_uint4(0u, 0u, 0u, 0u), o2 = o1;
        const bool fac = kg == 0 && (b & (SG - 1)) == 0;
        if (fac && t >= M) tokf[t * (nb / SG) + b / SG] = 1.f;
        if (t < M) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(Xq + t * K + b * KB + kg * 8));
            const float4 *dc = reinterpret_cast<const float4 *>(dx + t * nb + (b & ~(SG - 1)));
            const int st = chunk_exp(max8_f32(__ldg(dc), __ldg(dc + 1)), kTokExp);
            if (fac) tokf[t * (nb / SG) + b / SG] = exp2i(-st);
            const float d = __ldg(dx + t * nb + b) * exp2i(st);  // exact (both normal or zero)
            float e[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                e[j] = d * static_cast<float>(static_cast<int8_t>(v.x >> (8 * j)));
                e[j + 4] = d * static_cast<float>(static_cast<int8_t>(v.y >> (8 * j)));
            }
            uint32_t w1[4], w2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // word i holds elements (i, i+4)
                float r1a, r1b, r2a, r2b;
                w1[i] = split_h2(e[i], e[i + 4], r1a, r1b);
                w2[i] = split_h2(r1a, r1b, r2a, r2b);
            }
            o1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            o2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
        }
        uint4 *dst = Xh + chunk * (A_BYTES / 16) + within;
        dst[0] = o1;
        dst[APIECE / 16] = o2;
    }
}

// Weight pieces of one 8-element group: nibbles of w (element order) and
// the block's scale d = d_w * 2^u_r as f16x2 {d, d} (and -d) -> B1 and -B2
// chunks (16 bytes each, word i = elements (i, i+4)), all in packed f16:
// pair i is OR-ed into the f16 pattern of 1024 (exact 1024 + q*16^(i%2),
// after a shift by 8 for i >= 2), one FMA gives q - 8 exactly, B1 =
// RN(d * (q - 8)) and -B2 = B1 - d * (q - 8) by one FMA, exact because
// d * (q - 8) has at most 14 significant bits (11 x 3), so the remainder
// fits in f16 (in the normal range; d is at most 2^12, so |B1| <= 2^15).
// The MMA of the second piece negates B (kNegB).
__device__ __forceinline__ void nib8_split(uint32_t w, uint32_t d2, uint32_t nd2, uint4 &b1, uint4 &b2)
{
    asm("{\n"
        " .reg .b32 s, x0, x1, x2, x3, q0, q1, q2, q3, one, m1032, sixteenth, m72;\n"
        " mov.b32 one, 0x3C003C00;\n"        // 1
        " mov.b32 m1032, 0xE408E408;\n"      // -1032
        " mov.b32 sixteenth, 0x2C002C00;\n"  // 1/16
        " mov.b32 m72, 0xD480D480;\n"        // -72
        " shr.u32 s, %8, 8;\n"
        " lop3.b32 x0, %8, 0x000F000F, 0x64006400, 0xEA;\n"
        " lop3.b32 x1, %8, 0x00F000F0, 0x64006400, 0xEA;\n"
        " lop3.b32 x2, s, 0x000F000F, 0x64006400, 0xEA;\n"
        " lop3.b32 x3, s, 0x00F000F0, 0x64006400, 0xEA;\n"
        " fma.rn.f16x2 q0, x0, one, m1032;\n"  // x * 1 - 1032
        " fma.rn.f16x2 q1, x1, sixteenth, m72;\n"  // x / 16 - 72
        " fma.rn.f16x2 q2, x2, one, m1032;\n"
        " fma.rn.f16x2 q3, x3, sixteenth, m72;\n"
        " mul.rn.f16x2 %0, q0, %9;\n"
        " mul.rn.f16x2 %1, q1, %9;\n"
        " mul.rn.f16x2 %2, q2, %9;\n"
        " mul.rn.f16x2 %3, q3, %9;\n"
        " fma.rn.f16x2 %4, q0, %10, %0;\n"
        " fma.rn.f16x2 %5, q1, %10, %1;\n"
        " fma.rn.f16x2 %6, q2, %10, %2;\n"
        " fma.rn.f16x2 %7, q3, %10, %3;\n"
        "}"
        // every output is written before the last read of an input: early-clobber
        : "=&r"(b1.x), "=&r"(b1.y), "=&r"(b1.z), "=&r"(b1.w), "=&r"(b2.x), "=&r"(b2.y), "=&r"(b2.z), "=&r"(b2.w)
        : "r"(w), "r"(d2), "r"(nd2));
}

struct Work {
    int ntm, ntiles, nb;
};
__device__ __forceinline__ void tile_origin(const Work &w, int tile, int &t0, int &r0)
{
    const int tr = tile / w.ntm;
    t0 = (tile - tr * w.ntm) * TM;
    r0 = tr * TN;
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_split(const uint8_t *__restrict__ Xh, const __grid_constant__ CUtensorMap mapB,
                 const __grid_constant__ CUtensorMap mapW, const float *__restrict__ tokf,
                 float *__restrict__ Y, int rows, int K, int M, int *__restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_afull = sbase + OFF_BAR, bar_opempty = bar_afull + 8 * S, bar_full = bar_opempty + 8 * S;
    const uint32_t bar_rfull = bar_full + 8 * S, bar_rempty = bar_rfull + 8 * RAW;
    const uint32_t bar_cfull = bar_rempty + 8 * RAW, bar_cempty = bar_cfull + 8 * NACC;
    const uint32_t bar_sfull = bar_cempty + 8 * NACC, bar_sempty = bar_sfull + 8 * STG;
    const uint32_t bar_srdy = bar_sempty + 8 * STG;
    const uint32_t bar_drain = bar_srdy + 8 * NSR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    Work w;
    w.nb = K / KB;
    w.ntm = (M + TM - 1) / TM;
    w.ntiles = w.ntm * ((rows + TN - 1) / TN);
    const int my_tiles = (w.ntiles > static_cast<int>(blockIdx.x))
                             ? (w.ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const int nblocks = my_tiles * w.nb;  // the host checks that this fits an int

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(bar_afull + 8 * i, 1);
            mbar_init(bar_opempty + 8 * i, 1);
            mbar_init(bar_full + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < RAW; ++i) {
            mbar_init(bar_rfull + 8 * i, 1);
            mbar_init(bar_rempty + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(bar_cfull + 8 * i, 1);
            mbar_init(bar_cempty + 8 * i, RO_WARPS);
        }
        for (int i = 0; i < STG; ++i) {
            mbar_init(bar_sfull + 8 * i, 1);
            mbar_init(bar_sempty + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NSR; ++i) mbar_init(bar_srdy + 8 * i, CONV_WARPS);
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
        // ------------------------------------------------ nibble and scale tile loads
        if (lane == 0) {
            int tile = static_cast<int>(blockIdx.x), b = 0, t0, r0;
            tile_origin(w, tile, t0, r0);
            int rs = 0, nr = 0, gi = 0;
            uint32_t rph = 0;
            for (int gb = 0; gb < nblocks; ++gb) {
                if ((b & (SG - 1)) == 0) {
                    const int sg = gi & (STG - 1);
                    if (!wait_bounded(bar_sempty + 8 * sg, (static_cast<uint32_t>(gi / STG) & 1u) ^ 1u, abort, status))
                        break;
                    mbar_expect_tx(bar_sfull + 8 * sg, STW_BYTES);
                    tma_load_2d(sbase + OFF_STILE + sg * STW_BYTES, &mapW, b, r0, bar_sfull + 8 * sg);
                    ++gi;
                }
                if (!wait_bounded(bar_rempty + 8 * rs, rph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_rfull + 8 * rs, RB_BYTES);
                tma_load_2d(sbase + OFF_RAW + rs * RB_BYTES, &mapB, b * 16, r0, bar_rfull + 8 * rs);
                ++nr;
                if (++rs == RAW) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++b == w.nb) {
                    b = 0;
                    tile += static_cast<int>(gridDim.x);
                    tile_origin(w, tile, t0, r0);
                }
            }
            // No load may still be landing in shared memory when the CTA exits
            // (relevant only after an abort: normally every load has been consumed).
            volatile int no_abort = 0;
            for (int g = (nr > RAW ? nr - RAW : 0); g < nr; ++g)
                wait_bounded(bar_rfull + 8 * (g % RAW), static_cast<uint32_t>((g / RAW) & 1), &no_abort, status);
            for (int g = (gi > STG ? gi - STG : 0); g < gi; ++g)
                wait_bounded(bar_sfull + 8 * (g % STG), static_cast<uint32_t>((g / STG) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == ACOPY_WARP) {
        // ------------------------------------------------ A operand copies
        if (lane == 0) {
            int tile = static_cast<int>(blockIdx.x), b = 0, t0, r0;
            tile_origin(w, tile, t0, r0);
            int s = 0, na = 0;
            uint32_t sph = 0;
            for (int gb = 0; gb < nblocks; ++gb) {
                if (!wait_bounded(bar_opempty + 8 * s, sph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_afull + 8 * s, A_BYTES);
                bulk_load(sbase + OFF_A + s * A_BYTES,
                          Xh + (static_cast<size_t>(t0 / TM) * w.nb + b) * static_cast<size_t>(A_BYTES), A_BYTES,
                          bar_afull + 8 * s);
                ++na;
                if (++s == S) {
                    s = 0;
                    sph ^= 1u;
                }
                if (++b == w.nb) {
                    b = 0;
                    tile += static_cast<int>(gridDim.x);
                    tile_origin(w, tile, t0, r0);
                }
            }
            volatile int no_abort = 0;
            for (int g = (na > S ? na - S : 0); g < na; ++g)
                wait_bounded(bar_afull + 8 * (g % S), static_cast<uint32_t>((g / S) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t sph = 0;
            for (int gb = 0; gb < nblocks; ++gb) {
                const int ci = gb / SG, acc = ci & (NACC - 1);  // chunk, its accumulator
                const bool cfirst = (gb & (SG - 1)) == 0;
                if (!wait_bounded(bar_afull + 8 * s, sph, abort, status)) break;
                if (!wait_bounded(bar_full + 8 * s, sph, abort, status)) break;
                if (cfirst &&
                    !wait_bounded(bar_cempty + 8 * acc, (static_cast<uint32_t>(ci / NACC) & 1u) ^ 1u, abort, status))
                    break;
                tc_fence_after();
                const uint32_t a0 = sbase + OFF_A + s * A_BYTES, b0 = sbase + OFF_B + s * B_BYTES;
                const uint32_t d = tmem + acc * ACC_STRIDE;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint32_t ka = a0 + ks * 256, kb = b0 + ks * 256;
                    const uint64_t A1 = smem_desc(ka, 128, 512), A2 = smem_desc(ka + APIECE, 128, 512);
                    const uint64_t B1 = smem_desc(kb, 128, 512), B2 = smem_desc(kb + BPIECE, 128, 512);
                    mma_f16(d, A1, B1, kIdesc, (cfirst && ks == 0) ? 0u : 1u);
                    mma_f16(d, A1, B2, kIdesc | kNegB, 1u);
                    mma_f16(d, A2, B1, kIdesc, 1u);
                }
                mma_commit(bar_opempty + 8 * s);
                if ((gb & (SG - 1)) == SG - 1) mma_commit(bar_cfull + 8 * acc);
                if (++s == S) {
                    s = 0;
                    sph ^= 1u;
                }
            }
            // every issued MMA has completed before tensor memory is released
            mma_commit(bar_drain);
            wait_bounded(bar_drain, 0u, abort, status);
        }
        __syncwarp();
    } else if (warp < RO_WARPS) {
        // ------------------------------------------------ read-out warps
        const int q = warp & 3;  // TMEM lane quarter
        const int c0 = (warp >> 2) * EPI_COLS;
        bool ok = true;
        // Chunks hold SG consecutive blocks of one tile (nb % SG == 0).
        const int cpt = w.nb / SG;  // chunks per tile
        const int nchunks = nblocks / SG;
        float acc[EPI_COLS];  // written first by each tile's first chunk
        // 2^-s_t of this lane's token, loaded one chunk ahead
        auto token_factor = [&](int c) -> float {
            int t0, r0;
            tile_origin(w, static_cast<int>(blockIdx.x) + (c / cpt) * static_cast<int>(gridDim.x), t0, r0);
            return __ldg(tokf + static_cast<size_t>(t0 + q * 32 + lane) * cpt + c % cpt);
        };
        float ft_next = nchunks > 0 ? token_factor(0) : 1.f;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int ab = c & (NACC - 1);
            const int ct = c % cpt;  // chunk within its tile
            const float ft = ft_next;
            if (c + 1 < nchunks) ft_next = token_factor(c + 1);
            // 2^-u_r of the chunk's rows, written by the converters at its start
            ok = wait_warp(bar_srdy + 8 * (c & (NSR - 1)), static_cast<uint32_t>(c / NSR) & 1u, abort, status);
            if (!ok) break;
            const float *sr = reinterpret_cast<const float *>(smem + OFF_SR + (c & (NSR - 1)) * SR_BYTES) + c0;
            ok = wait_warp(bar_cfull + 8 * ab, static_cast<uint32_t>(c / NACC) & 1u, abort, status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + ab * ACC_STRIDE + c0;
#pragma unroll
            for (int part = 0; part < EPI_COLS / 16; ++part) {
                float d[16];
                tmem_ld16(taddr + part * 16, d);
                if (part == EPI_COLS / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_cempty + 8 * ab);
                }
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    const float4 f4 = *reinterpret_cast<const float4 *>(sr + part * 16 + e);
                    const float2 f01 = __fmul2_rn(make_float2(ft, ft), make_float2(f4.x, f4.y));  // exact
                    const float2 f23 = __fmul2_rn(make_float2(ft, ft), make_float2(f4.z, f4.w));
                    float2 v01, v23;
                    if (ct != 0) {
                        v01 = __ffma2_rn(make_float2(d[e], d[e + 1]), f01,
                                         make_float2(acc[part * 16 + e], acc[part * 16 + e + 1]));
                        v23 = __ffma2_rn(make_float2(d[e + 2], d[e + 3]), f23,
                                         make_float2(acc[part * 16 + e + 2], acc[part * 16 + e + 3]));
                    } else {
                        v01 = __fmul2_rn(make_float2(d[e], d[e + 1]), f01);
                        v23 = __fmul2_rn(make_float2(d[e + 2], d[e + 3]), f23);
                    }
                    acc[part * 16 + e] = v01.x;
                    acc[part * 16 + e + 1] = v01.y;
                    acc[part * 16 + e + 2] = v23.x;
                    acc[part * 16 + e + 3] = v23.y;
                }
            }
            if (ct == cpt - 1) {
                int t0, r0;
                tile_origin(w, static_cast<int>(blockIdx.x) + (c / cpt) * static_cast<int>(gridDim.x), t0, r0);
                const int t = t0 + q * 32 + lane;
                if (t < M) {
                    float *yrow = Y + static_cast<size_t>(t) * rows + r0 + c0;
                    const int nvalid = rows - (r0 + c0);
                    const bool vec = (rows & 3) == 0;
#pragma unroll
                    for (int cc = 0; cc < EPI_COLS; cc += 4) {
                        if (vec && cc + 4 <= nvalid) {
                            *reinterpret_cast<float4 *>(yrow + cc) =
                                make_float4(acc[cc], acc[cc + 1], acc[cc + 2], acc[cc + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (cc + e < nvalid) yrow[cc + e] = acc[cc + e];
                        }
                    }
                }
            }
        }
    } else if (warp < CONV0 + CONV_WARPS) {
        // ------------------------------------------------ converter warps
        // warp v: nibble words 2h, 2h+1 (h = v % 2) of rows 32*(v/2) + 64k + lane,
        // so the 16-byte stores of 8 consecutive lanes fall on distinct bank groups
        const int v = warp - CONV0, h = v & 1;
        int crow[CROWS];
#pragma unroll
        for (int k = 0; k < CROWS; ++k) crow[k] = 32 * (v >> 1) + 64 * k + lane;
        bool ok = true;
        float wsc[CROWS];  // 2^u_r of each converted row for the current chunk
#pragma unroll
        for (int k = 0; k < CROWS; ++k) wsc[k] = 1.f;
        for (int g = 0; g < nblocks && ok; ++g) {
            const int s = g & (S - 1), rs = g & (RAW - 1), sg = (g / SG) & (STG - 1);
            // the stage's previous block (g - S) must be done in the tensor core
            if (g >= S) ok = wait_warp(bar_opempty + 8 * s, static_cast<uint32_t>(g / S - 1) & 1u, abort, status);
            if (ok && (g & (SG - 1)) == 0)
                ok = wait_warp(bar_sfull + 8 * sg, static_cast<uint32_t>(g / (SG * STG)) & 1u, abort, status);
            if (ok) ok = wait_warp(bar_rfull + 8 * rs, static_cast<uint32_t>(g / RAW) & 1u, abort, status);
            if (!ok) break;
            const uint8_t *stile = smem + OFF_STILE + sg * STW_BYTES;
            const int cg = g / SG;  // chunk of this block
            if ((g & (SG - 1)) == 0) {
                // 2^u_r of each row for the chunk (rows past the end load zeros: 1),
                // and 2^-u_r into the chunk's row-factor slot for the read-out
                float *srs = reinterpret_cast<float *>(smem + OFF_SR + (cg & (NSR - 1)) * SR_BYTES);
#pragma unroll
                for (int k = 0; k < CROWS; ++k) {
                    const int u =
                        chunk_exp(max8_f16(*reinterpret_cast<const uint4 *>(stile + crow[k] * 16)), kRowExp);
                    wsc[k] = exp2i(u);
                    if (h == 0) srs[crow[k]] = exp2i(-u);
                }
            }
            uint8_t *stage = smem + OFF_B + s * B_BYTES;
            const uint8_t *raw = smem + OFF_RAW + rs * RB_BYTES;
#pragma unroll
            for (int k = 0; k < CROWS; ++k) {
                const uint16_t dwb = reinterpret_cast<const uint16_t *>(stile)[crow[k] * SG + (g & (SG - 1))];
                // d_w * 2^u_r: exact in f32, and in f16 down to 2^-14 (at most 2^12)
                const uint32_t dh =
                    __half_as_ushort(__float2half_rn(__half2float(__ushort_as_half(dwb)) * wsc[k]));
                const uint32_t dw = dh | (dh << 16), ndw = dw ^ 0x80008000u;
                const uint2 nv = *reinterpret_cast<const uint2 *>(raw + crow[k] * 16 + h * 8);
                uint8_t *dst = stage + op_off(crow[k], 2 * h);
                uint4 b1, b2;
                nib8_split(nv.x, dw, ndw, b1, b2);
                *reinterpret_cast<uint4 *>(dst) = b1;
                *reinterpret_cast<uint4 *>(dst + BPIECE) = b2;
                nib8_split(nv.y, dw, ndw, b1, b2);
                *reinterpret_cast<uint4 *>(dst + 128) = b1;
                *reinterpret_cast<uint4 *>(dst + BPIECE + 128) = b2;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_full + 8 * s);
                mbar_arrive(bar_rempty + 8 * rs);
                if ((g & (SG - 1)) == 0) mbar_arrive(bar_srdy + 8 * (cg & (NSR - 1)));
                if ((g & (SG - 1)) == SG - 1) mbar_arrive(bar_sempty + 8 * sg);
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

// ---------------------------------------------------------------- the CTA-pair kernel
// Same operands and chunking as k_gemm_split, with one M = 256 MMA per CTA
// pair (cta_group::2): a cluster of two CTAs takes 256-token x 192-row
// tiles; CTA rank c holds tokens 128c.. of the tile as its half of A (and of
// D in its tensor memory) and rows 96c.. as its half of B, so each CTA
// converts 96 rows per block instead of 192 and the tensor core reads half
// of B from each SM.  Rank 0 issues the MMAs; the peer's converters and
// read-out warps arrive on rank 0's barriers, and rank 0's commits signal
// both CTAs.
namespace pair {
constexpr int HN = TN / 2;               // rows of B per CTA
constexpr int PS = 6;                    // operand stages (A half + B half = 28 KB each)
constexpr int PS2 = PS / 2;              // pair stages: one barrier phase per two blocks
constexpr int BPIECE = HN * KB * 2;      // 6144: one f16 piece of this CTA's B half
constexpr int B_BYTES = 2 * BPIECE;      // 12288
constexpr int RBP_BYTES = HN * 32;       // 3072: nibbles of two blocks (TMA box 32 x 96)
constexpr int RAWP = 4;                  // raw stages (block pairs)
constexpr int STW_BYTES = TN * SG * 2;   // 3072: d_w of all 192 rows (TMA box 8 x 192)
constexpr int CONV_WARPS = 6;            // one row of one block (16 B of nibbles) per lane per block pair
constexpr int CONV0 = RO_WARPS;
constexpr int TMA_WARP = RO_WARPS + CONV_WARPS;
constexpr int MMA_WARP = TMA_WARP + 1;
constexpr int ACOPY_WARP = TMA_WARP + 2;
constexpr int NTHREADS = (ACOPY_WARP + 1) * 32;  // 672

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + PS * A_BYTES;
constexpr int OFF_RAW = OFF_B + PS * B_BYTES;
constexpr int OFF_STILE = OFF_RAW + RAWP * RBP_BYTES;
constexpr int OFF_SR = OFF_STILE + STG * STW_BYTES;
constexpr int OFF_BAR = OFF_SR + NSR * SR_BYTES;
constexpr int N_BARS = 3 * PS2 + 2 * RAWP + 2 * NACC + 2 * STG + NSR + 1;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int OFF_RELAY = (OFF_MISC + 16 + 15) / 16 * 16;  // PS2 x 16 B: rank 0's landing slots of the relay copies
constexpr int RELAY_BYTES = 16;
constexpr int SMEM_BYTES = OFF_RELAY + PS2 * RELAY_BYTES;
static_assert(OFF_B % 1024 == 0 && OFF_RAW % 1024 == 0 && OFF_STILE % 128 == 0 && OFF_SR % 16 == 0 &&
                  OFF_BAR % 8 == 0 && SMEM_BYTES <= 232448,
              "shared memory layout");
static_assert(CONV_WARPS * 32 == 2 * HN && CONV_WARPS * 32 == TN, "converter threads: 2 per B row (one per block of a pair), 1 per tile row");
static_assert(PS % 2 == 0 && SG % 2 == 0, "block pairs never straddle a stage wrap, a chunk or a tile (nb % 8 == 0)");
constexpr uint32_t kIdesc = idesc_f16(2 * TM, TN, false);  // M = 256 over the pair

struct Work {
    int ntm2, ntiles, nb;  // 256-token tiles, tiles, blocks per row
};
__device__ __forceinline__ void tile_origin(const Work &w, int tile, int &t0, int &r0)
{
    const int tr = tile / w.ntm2;
    t0 = (tile - tr * w.ntm2) * 2 * TM;
    r0 = tr * TN;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_pair(const uint8_t *__restrict__ Xh, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapW, const float *__restrict__ tokf, float *__restrict__ Y,
                int rows, int K, int M, int *__restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t sbase = smem_u32(smem);
    // full (rank 0): its converters, its A copy and the peer's relay bytes;
    // pfull (rank 1): its converters and its A copy, forwarded by the relay
    // (per pair stage: blocks 2p and 2p + 1 of the CTA's sequence, p = pair index)
    const uint32_t bar_pfull = sbase + OFF_BAR, bar_opempty = bar_pfull + 8 * PS2, bar_full = bar_opempty + 8 * PS2;
    const uint32_t bar_rfull = bar_full + 8 * PS2, bar_rempty = bar_rfull + 8 * RAWP;
    const uint32_t bar_cfull = bar_rempty + 8 * RAWP, bar_cempty = bar_cfull + 8 * NACC;
    const uint32_t bar_sfull = bar_cempty + 8 * NACC, bar_sempty = bar_sfull + 8 * STG;
    const uint32_t bar_srdy = bar_sempty + 8 * STG;
    const uint32_t bar_drain = bar_srdy + 8 * NSR;
    const uint32_t bar_mine = rank == 0 ? bar_full : bar_pfull;  // where this CTA's stage producers arrive
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    Work w;
    w.nb = K / KB;
    w.ntm2 = (M + 2 * TM - 1) / (2 * TM);
    w.ntiles = w.ntm2 * ((rows + TN - 1) / TN);
    const int cid = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);
    const int my_tiles = (w.ntiles > cid) ? (w.ntiles - 1 - cid) / ncl + 1 : 0;
    const int nblocks = my_tiles * w.nb;  // the same in both CTAs of the pair

    if (threadIdx.x == 0) {
        for (int i = 0; i < PS2; ++i) {
            mbar_init(bar_opempty + 8 * i, 1);
            // converters + the A copy's arrival (with its bytes); rank 0's full
            // also expects RELAY_BYTES from the peer's relay copy
            mbar_init(bar_full + 8 * i, CONV_WARPS + 1);
            mbar_init(bar_pfull + 8 * i, CONV_WARPS + 1);
        }
        for (int i = 0; i < RAWP; ++i) {
            mbar_init(bar_rfull + 8 * i, 1);
            mbar_init(bar_rempty + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(bar_cfull + 8 * i, 1);
            mbar_init(bar_cempty + 8 * i, 2 * RO_WARPS);  // rank 0's: both CTAs' read-out warps
        }
        for (int i = 0; i < STG; ++i) {
            mbar_init(bar_sfull + 8 * i, 1);
            mbar_init(bar_sempty + 8 * i, CONV_WARPS);
        }
        for (int i = 0; i < NSR; ++i) mbar_init(bar_srdy + 8 * i, CONV_WARPS);
        mbar_init(bar_drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MMA_WARP) {  // one warp of each CTA of the pair
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialized before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    if (warp == TMA_WARP) {
        // ------------------------------------------------ nibble (this CTA's 96 rows) and scale (192 rows) tiles
        if (lane == 0) {
            int tile = cid, b = 0, t0, r0;
            tile_origin(w, tile, t0, r0);
            int rs = 0, nr = 0, gi = 0;
            uint32_t rph = 0;
            for (int gb = 0; gb < nblocks; gb += 2) {
                if ((b & (SG - 1)) == 0) {
                    const int sg = gi & (STG - 1);
                    if (!wait_bounded(bar_sempty + 8 * sg, (static_cast<uint32_t>(gi / STG) & 1u) ^ 1u, abort, status))
                        break;
                    mbar_expect_tx(bar_sfull + 8 * sg, STW_BYTES);
                    tma_load_2d(sbase + OFF_STILE + sg * STW_BYTES, &mapW, b, r0, bar_sfull + 8 * sg);
                    ++gi;
                }
                if (!wait_bounded(bar_rempty + 8 * rs, rph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_rfull + 8 * rs, RBP_BYTES);
                tma_load_2d(sbase + OFF_RAW + rs * RBP_BYTES, &mapB, b * 16, r0 + static_cast<int>(rank) * HN,
                            bar_rfull + 8 * rs);
                ++nr;
                if (++rs == RAWP) {
                    rs = 0;
                    rph ^= 1u;
                }
                b += 2;
                if (b == w.nb) {
                    b = 0;
                    tile += ncl;
                    tile_origin(w, tile, t0, r0);
                }
            }
            volatile int no_abort = 0;
            for (int g = (nr > RAWP ? nr - RAWP : 0); g < nr; ++g)
                wait_bounded(bar_rfull + 8 * (g % RAWP), static_cast<uint32_t>((g / RAWP) & 1), &no_abort, status);
            for (int g = (gi > STG ? gi - STG : 0); g < gi; ++g)
                wait_bounded(bar_sfull + 8 * (g % STG), static_cast<uint32_t>((g / STG) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == ACOPY_WARP) {
        // ------------------------------------------------ this CTA's half of A
        if (lane == 0) {
            int tile = cid, b = 0, t0, r0;
            tile_origin(w, tile, t0, r0);
            int sp = 0, na = 0;
            uint32_t sph = 0;
            for (int gb = 0; gb < nblocks; gb += 2) {
                if (!wait_bounded<true>(bar_opempty + 8 * sp, sph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_mine + 8 * sp, 2 * A_BYTES);
                const size_t T = static_cast<size_t>(t0 / TM) + rank;  // 128-token tile
                const uint8_t *src = Xh + (T * w.nb + b) * static_cast<size_t>(A_BYTES);  // blocks b, b + 1
                bulk_load(sbase + OFF_A + 2 * sp * A_BYTES, src, A_BYTES, bar_mine + 8 * sp);
                bulk_load(sbase + OFF_A + (2 * sp + 1) * A_BYTES, src + A_BYTES, A_BYTES, bar_mine + 8 * sp);
                ++na;
                if (++sp == PS2) {
                    sp = 0;
                    sph ^= 1u;
                }
                b += 2;
                if (b == w.nb) {
                    b = 0;
                    tile += ncl;
                    tile_origin(w, tile, t0, r0);
                }
            }
            // no copy may still be landing when the CTA exits (after an abort the
            // stage's other arrivals may be missing: the waits then time out)
            volatile int no_abort = 0;
            for (int g = (na > PS2 ? na - PS2 : 0); g < na; ++g)
                wait_bounded<true>(bar_mine + 8 * (g % PS2), static_cast<uint32_t>((g / PS2) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issuer (rank 0)
        if (lane == 0 && rank == 0) {
            int sp = 0;
            uint32_t sph = 0;
            for (int gb = 0; gb < nblocks; gb += 2) {
                const int ci = gb / SG, acc = ci & (NACC - 1);
                const bool cfirst = (gb & (SG - 1)) == 0;
                if (!wait_bounded<true>(bar_full + 8 * sp, sph, abort, status)) break;
                if (cfirst && !wait_bounded<true>(bar_cempty + 8 * acc, (static_cast<uint32_t>(ci / NACC) & 1u) ^ 1u,
                                                  abort, status))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + acc * ACC_STRIDE;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t a0 = sbase + OFF_A + (2 * sp + j) * A_BYTES, b0 = sbase + OFF_B + (2 * sp + j) * B_BYTES;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint32_t ka = a0 + ks * 256, kb = b0 + ks * 256;
                        const uint64_t A1 = smem_desc(ka, 128, 512), A2 = smem_desc(ka + APIECE, 128, 512);
                        const uint64_t B1 = smem_desc(kb, 128, 512), B2 = smem_desc(kb + BPIECE, 128, 512);
                        mma_f16_pair(d, A1, B1, kIdesc, (cfirst && j == 0 && ks == 0) ? 0u : 1u);
                        mma_f16_pair(d, A1, B2, kIdesc | kNegB, 1u);
                        mma_f16_pair(d, A2, B1, kIdesc, 1u);
                    }
                }
                mma_commit_pair(bar_opempty + 8 * sp);
                if ((gb & (SG - 1)) == SG - 2) mma_commit_pair(bar_cfull + 8 * acc);
                if (++sp == PS2) {
                    sp = 0;
                    sph ^= 1u;
                }
            }
            // every issued MMA has completed before either CTA releases tensor memory
            mma_commit_pair(bar_drain);
        }
        if (lane == 0 && rank != 0) {
            // relay: once this CTA's B half (its converters) and A half (its
            // bulk copy) of a stage are in shared memory, a 16-byte copy into
            // rank 0's shared memory completes RELAY_BYTES of rank 0's full
            // barrier for the stage (an async-proxy signal: the thread does not
            // wait for it to land)
            const uint32_t full0 = mapa_shared(bar_full, 0);
            const uint32_t slot0 = mapa_shared(sbase + OFF_RELAY, 0);
            for (int p = 0; p < nblocks / 2; ++p) {
                const int sp = p % PS2;
                const uint32_t ph = static_cast<uint32_t>(p / PS2) & 1u;
                if (!wait_bounded(bar_pfull + 8 * sp, ph, abort, status)) break;
                asm volatile(
                    "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        slot0 + sp * RELAY_BYTES),
                    "r"(sbase + OFF_RELAY + sp * RELAY_BYTES), "r"(RELAY_BYTES), "r"(full0 + 8 * sp)
                    : "memory");
            }
            // every relay copy has landed before rank 0's MMAs of its stage were
            // issued, so the drain wait below also covers them
        }
        if (lane == 0) {
            volatile int no_abort = 0;
            wait_bounded<true>(bar_drain, 0u, &no_abort, status);
        }
        __syncwarp();
    } else if (warp < RO_WARPS) {
        // ------------------------------------------------ read-out warps (this CTA's 128 tokens)
        const int q = warp & 3;
        const int c0 = (warp >> 2) * EPI_COLS;
        const uint32_t cempty0 = mapa_shared(bar_cempty, 0);  // rank 0's barrier (for rank 1)
        bool ok = true;
        const int cpt = w.nb / SG;
        const int nchunks = nblocks / SG;
        float acc[EPI_COLS];
        auto token_factor = [&](int c) -> float {
            int t0, r0;
            tile_origin(w, cid + (c / cpt) * ncl, t0, r0);
            return __ldg(tokf + static_cast<size_t>(t0 + static_cast<int>(rank) * TM + q * 32 + lane) * cpt + c % cpt);
        };
        float ft_next = nchunks > 0 ? token_factor(0) : 1.f;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int ab = c & (NACC - 1);
            const int ct = c % cpt;
            const float ft = ft_next;
            if (c + 1 < nchunks) ft_next = token_factor(c + 1);
            ok = wait_warp(bar_srdy + 8 * (c & (NSR - 1)), static_cast<uint32_t>(c / NSR) & 1u, abort, status);
            if (!ok) break;
            const float *sr = reinterpret_cast<const float *>(smem + OFF_SR + (c & (NSR - 1)) * SR_BYTES) + c0;
            ok = wait_warp<true>(bar_cfull + 8 * ab, static_cast<uint32_t>(c / NACC) & 1u, abort, status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + ab * ACC_STRIDE + c0;
#pragma unroll
            for (int part = 0; part < EPI_COLS / 16; ++part) {
                float d[16];
                tmem_ld16(taddr + part * 16, d);
                if (part == EPI_COLS / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank == 0)
                            mbar_arrive(bar_cempty + 8 * ab);
                        else
                            mbar_arrive_cluster(cempty0 + 8 * ab);
                    }
                }
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    const float4 f4 = *reinterpret_cast<const float4 *>(sr + part * 16 + e);
                    const float2 f01 = __fmul2_rn(make_float2(ft, ft), make_float2(f4.x, f4.y));  // exact
                    const float2 f23 = __fmul2_rn(make_float2(ft, ft), make_float2(f4.z, f4.w));
                    float2 v01, v23;
                    if (ct != 0) {
                        v01 = __ffma2_rn(make_float2(d[e], d[e + 1]), f01,
                                         make_float2(acc[part * 16 + e], acc[part * 16 + e + 1]));
                        v23 = __ffma2_rn(make_float2(d[e + 2], d[e + 3]), f23,
                                         make_float2(acc[part * 16 + e + 2], acc[part * 16 + e + 3]));
                    } else {
                        v01 = __fmul2_rn(make_float2(d[e], d[e + 1]), f01);
                        v23 = __fmul2_rn(make_float2(d[e + 2], d[e + 3]), f23);
                    }
                    acc[part * 16 + e] = v01.x;
                    acc[part * 16 + e + 1] = v01.y;
                    acc[part * 16 + e + 2] = v23.x;
                    acc[part * 16 + e + 3] = v23.y;
                }
            }
            if (ct == cpt - 1) {
                int t0, r0;
                tile_origin(w, cid + (c / cpt) * ncl, t0, r0);
                const int t = t0 + static_cast<int>(rank) * TM + q * 32 + lane;
                if (t < M) {
                    float *yrow = Y + static_cast<size_t>(t) * rows + r0 + c0;
                    const int nvalid = rows - (r0 + c0);
                    const bool vec = (rows & 3) == 0;
#pragma unroll
                    for (int cc = 0; cc < EPI_COLS; cc += 4) {
                        if (vec && cc + 4 <= nvalid) {
                            *reinterpret_cast<float4 *>(yrow + cc) =
                                make_float4(acc[cc], acc[cc + 1], acc[cc + 2], acc[cc + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (cc + e < nvalid) yrow[cc + e] = acc[cc + e];
                        }
                    }
                }
            }
        }
    } else if (warp < CONV0 + CONV_WARPS) {
        // ------------------------------------------------ converter warps (this CTA's 96 rows)
        // warp v: all four nibble words of half-tile row 32*(v/2) + lane in block
        // g + h (h = v % 2) of each pair g, g + 1; for the read-out, the chunk
        // factor of tile row 32*v + lane
        const int v = warp - CONV0, h = v & 1;
        const int crow = 32 * (v >> 1) + lane;                   // row of this CTA's B half
        const int trow = static_cast<int>(rank) * HN + crow;    // the same row in the tile
        const int frow = 32 * v + lane;                          // row whose factor this thread writes
        bool ok = true;
        float wsc = 1.f;
        for (int g = 0; g < nblocks && ok; g += 2) {  // blocks g, g + 1: stages s, s + 1
            const int p = g >> 1, sp = p % PS2, s = 2 * sp, rs = p & (RAWP - 1), sg = (g / SG) & (STG - 1);
            if (p >= PS2)
                ok = wait_warp<true>(bar_opempty + 8 * sp, static_cast<uint32_t>(p / PS2 - 1) & 1u, abort, status);
            if (ok && (g & (SG - 1)) == 0)
                ok = wait_warp(bar_sfull + 8 * sg, static_cast<uint32_t>(g / (SG * STG)) & 1u, abort, status);
            if (ok) ok = wait_warp(bar_rfull + 8 * rs, static_cast<uint32_t>(p / RAWP) & 1u, abort, status);
            if (!ok) break;
            const uint8_t *stile = smem + OFF_STILE + sg * STW_BYTES;
            const int cg = g / SG;
            if ((g & (SG - 1)) == 0) {
                wsc = exp2i(chunk_exp(max8_f16(*reinterpret_cast<const uint4 *>(stile + trow * 16)), kRowExp));
                const int uf = chunk_exp(max8_f16(*reinterpret_cast<const uint4 *>(stile + frow * 16)), kRowExp);
                reinterpret_cast<float *>(smem + OFF_SR + (cg & (NSR - 1)) * SR_BYTES)[frow] = exp2i(-uf);
            }
            // d_w * 2^u_r of block g + h: exact in f32, and in f16 down to 2^-14 (at most 2^12)
            const uint16_t dwb = reinterpret_cast<const uint16_t *>(stile)[trow * SG + (g & (SG - 1)) + h];
            const uint32_t dh = __half_as_ushort(__float2half_rn(__half2float(__ushort_as_half(dwb)) * wsc));
            const uint32_t dw = dh | (dh << 16), ndw = dw ^ 0x80008000u;
            const uint4 nv = *reinterpret_cast<const uint4 *>(smem + OFF_RAW + rs * RBP_BYTES + crow * 32 + h * 16);
            uint8_t *dst = smem + OFF_B + (s + h) * B_BYTES + op_off(crow, 0);
            uint4 b1, b2;
            nib8_split(nv.x, dw, ndw, b1, b2);
            *reinterpret_cast<uint4 *>(dst) = b1;
            *reinterpret_cast<uint4 *>(dst + BPIECE) = b2;
            nib8_split(nv.y, dw, ndw, b1, b2);
            *reinterpret_cast<uint4 *>(dst + 128) = b1;
            *reinterpret_cast<uint4 *>(dst + BPIECE + 128) = b2;
            nib8_split(nv.z, dw, ndw, b1, b2);
            *reinterpret_cast<uint4 *>(dst + 256) = b1;
            *reinterpret_cast<uint4 *>(dst + BPIECE + 256) = b2;
            nib8_split(nv.w, dw, ndw, b1, b2);
            *reinterpret_cast<uint4 *>(dst + 384) = b1;
            *reinterpret_cast<uint4 *>(dst + BPIECE + 384) = b2;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0 && v == 0)
                    mbar_expect_tx(bar_full + 8 * sp, RELAY_BYTES);  // arrive + the peer's relay bytes
                else
                    mbar_arrive(bar_mine + 8 * sp);
                mbar_arrive(bar_rempty + 8 * rs);
                if ((g & (SG - 1)) == 0) mbar_arrive(bar_srdy + 8 * (cg & (NSR - 1)));
                if ((g & (SG - 1)) == SG - 2) mbar_arrive(bar_sempty + 8 * sg);
            }
        }
    }

    tc_fence_before();
    cluster_sync_all();  // no remote arrive or MMA operand read is still pending on either CTA
    pdl_launch_dependents();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}
}  // namespace pair

}  // namespace tcs

// ---------------------------------------------------------------- host side
// Workspace: the A chunks, then the token factors f32 [ntm * 128][K / 256],
// with ntm = the number of 128-token tiles rounded up to even (the pair
// kernel takes 256 tokens per tile; the pre-pass zero-fills the padding).
static int split_ntm(int M) { return 2 * ((M + 2 * tcs::TM - 1) / (2 * tcs::TM)); }
static size_t split_chunks_bytes(int K, int M)
{
    return static_cast<size_t>(split_ntm(M)) * static_cast<size_t>(K / tcs::KB) * tcs::A_BYTES;
}
size_t gemm_split_workspace_bytes(int K, int M)
{
    if (!gemm_split_supported(K) || M < 1) return 0;
    return split_chunks_bytes(K, M) +
           static_cast<size_t>(split_ntm(M)) * tcs::TM * static_cast<size_t>(K / (tcs::KB * tcs::SG)) * 4;
}

bool gemm_split_supported(int K) { return K >= 256 && K % 256 == 0; }

// Clusters of two k_gemm_pair CTAs that can be resident at once (0 if none).
static int pair_clusters()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] != 0) return cache[dev] > 0 ? cache[dev] : 0;
    if (ctas_per_sm(reinterpret_cast<const void *>(tcs::pair::k_gemm_pair), tcs::pair::NTHREADS,
                    tcs::pair::SMEM_BYTES) <= 0) {
        cache[dev] = -1;
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(sm_count()));
    cfg.blockDim = dim3(tcs::pair::NTHREADS);
    cfg.dynamicSmemBytes = tcs::pair::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tcs::pair::k_gemm_pair, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        cache[dev] = -1;
        return 0;
    }
    cache[dev] = n;
    return n;
}

int launch_gemm_split(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes,
                      int rows, int K, int M, cudaStream_t s)
{
    if (!gemm_split_supported(K)) return GQ_ERR_SHAPE;
    const int nb = K / 32;
    const size_t need = gemm_split_workspace_bytes(K, M);
    if (need == 0) return GQ_ERR_SHAPE;
    if (ws_bytes < need) return GQ_ERR_WORKSPACE;
    // two CTAs per tile when there are at least two 128-token tiles (measured
    // at M = 32 on 21504 x 5376 weights: pairs 141 us, one CTA 125 us per step)
    const bool use_pair = M > tcs::TM && pair_clusters() > 0;
    const int tm = use_pair ? 2 * tcs::TM : tcs::TM;
    const long long ntiles_ll = static_cast<long long>((M + tm - 1) / tm) * ((rows + tcs::TN - 1) / tcs::TN);
    if (ntiles_ll * nb > 0x7FFFFFFFll) return GQ_ERR_SHAPE;  // per-CTA block counts are ints
    const int ntiles = static_cast<int>(ntiles_ll);
    const uint8_t *nib = static_cast<const uint8_t *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb * 16);
    CUtensorMap mapB, mapW;
    if (!make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, nib, static_cast<uint64_t>(nb) * 16,
                  static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 16, use_pair ? 32 : 16,
                  use_pair ? tcs::pair::HN : tcs::TN) ||
        !make_map(&mapW, CU_TENSOR_MAP_DATA_TYPE_UINT16, dsc, static_cast<uint64_t>(nb), static_cast<uint64_t>(rows),
                  static_cast<uint64_t>(nb) * 2, tcs::SG, tcs::TN))
        return GQ_ERR_CUDA;

    // activation codes x scales -> f16 operand pieces
    const size_t chunks_bytes = split_chunks_bytes(K, M);
    float *tokf = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + chunks_bytes);
    const long long npieces = static_cast<long long>(chunks_bytes / tcs::A_BYTES) * 512;
    long long pgrid = (npieces + 255) / 256;
    const long long pmax = static_cast<long long>(sm_count()) * 8;
    if (pgrid > pmax) pgrid = pmax;
    int rc = status_from(launch_pdl(tcs::k_xq_split, dim3(static_cast<unsigned>(pgrid)), dim3(256), 0, s, Xq, dx,
                                    static_cast<uint4 *>(ws), tokf, K, M, npieces));
    if (rc != GQ_OK) return rc;

    if (use_pair) {
        int ncl = pair_clusters();
        if (ncl > ntiles) ncl = ntiles;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * static_cast<unsigned>(ncl));
        cfg.blockDim = dim3(tcs::pair::NTHREADS);
        cfg.dynamicSmemBytes = tcs::pair::SMEM_BYTES;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return status_from(cudaLaunchKernelEx(&cfg, tcs::pair::k_gemm_pair, static_cast<const uint8_t *>(ws), mapB,
                                              mapW, static_cast<const float *>(tokf), Y, rows, K, M,
                                              status_word()));
    }
    const int occ = ctas_per_sm(reinterpret_cast<const void *>(tcs::k_gemm_split), tcs::NTHREADS, tcs::SMEM_BYTES);
    if (occ <= 0) return GQ_ERR_CUDA;
    int grid = sm_count();
    if (grid > ntiles) grid = ntiles;
    return status_from(launch_pdl(tcs::k_gemm_split, dim3(grid), dim3(tcs::NTHREADS),
                                  static_cast<size_t>(tcs::SMEM_BYTES), s, static_cast<const uint8_t *>(ws), mapB,
                                  mapW, static_cast<const float *>(tokf), Y, rows, K, M, status_word()));
}

}  // namespace gq
