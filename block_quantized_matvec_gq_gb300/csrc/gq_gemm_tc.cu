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
// Two kernels:
//   k_xq_to_ops  converts the activation codes once into f16 operand chunks
//                in the caller's workspace: one 8 KB chunk per (128-token
//                tile, 32-block), already in the UMMA K-major layout, so the
//                GEMM copies A with one bulk copy per block and never
//                converts it (A is reused by every weight tile).
//   k_gemm_q8act_tc, one 448-thread CTA per SM, persistent over 128-token x
//                192-row tiles, two accumulator buffers in TMEM:
//   warps 0-11  workers.  For block g: wait for its D, tcgen05.ld it (warp w
//               owns TMEM lanes 32*(w%4).. and 64 of the 192 columns), fold it
//               into the f32 accumulators, release the D buffer; then convert
//               the weight nibbles of block g+S into the f16 operand stage
//               the MMA of block g has finished with (two fixed 8-element
//               groups per thread) and stage its scales.
//   warp 12     one lane issues the TMA loads of the 192 x 16 B weight
//               nibbles of each block into an RAW-deep ring and, when K is a
//               multiple of 256, every 8 blocks the scale tiles of the next 8
//               blocks (d_w fp16 8 x 192, dx f32 8 x 128) into a 2-deep ring,
//               so the workers read scales from shared memory, never from
//               global memory inside the loop.
//   warp 13     one lane issues 2 x (M128 N192 K16) MMAs per block; the warp
//               owns the TMEM allocation.
//   warp 14     one lane issues the bulk copy of each block's A chunk into
//               its operand stage once the MMA has released the stage (its
//               own warp, so nibble loads never queue behind these waits).
// Tile and block coordinates advance incrementally (no integer division in
// the loops).
// Every mbarrier wait is bounded: on timeout the kernel records
// GQ_ERR_TIMEOUT in the device status word, every role leaves its loop, TMEM
// is released and the kernel returns.
#include "gq_tc.cuh"

namespace gq {
namespace tc {

using namespace tcu;

constexpr int TM = 128;  // tokens per tile (MMA M, TMEM lanes)
constexpr int TN = 192;  // weight rows per tile (MMA N, TMEM columns)
constexpr int KB = 32;   // K per quantization block
constexpr int S = 8;     // operand stages
constexpr int SR = 2 * S;  // scale stages
constexpr int RAW = 8;   // raw nibble stages (8 blocks of lead over the conversion)
constexpr int WORK_WARPS = 12;  // 4 TMEM lane quarters x 3 column groups
constexpr int NWORK = WORK_WARPS * 32;
constexpr int TMA_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr int ACOPY_WARP = 14;
constexpr int NTHREADS = 15 * 32;  // 480: up to 128 registers per thread
constexpr int EPI_COLS = TN / (WORK_WARPS / 4);  // 64
constexpr int NDBUF = 2;     // TMEM accumulator buffers (192 of 256 columns each)
constexpr int TMEM_COLS = 512;
constexpr int DBUF = 256;  // TMEM column offset between D buffers
constexpr uint32_t kIdesc = idesc_f16(TM, TN, false);  // f16 operands (exact small integers)

constexpr int A_BYTES = TM * KB * 2;  // 8192: f16 operand A (one workspace chunk)
constexpr int B_BYTES = TN * KB * 2;  // 12288: f16 operand B
constexpr int RB_BYTES = TN * 16;     // 3072: nibbles (TMA box 16 x 192)
constexpr int SCL_BYTES = (TM + TN) * 4;
constexpr int SG = 8;                 // blocks per scale tile
constexpr int STG = 2;                // scale tile stages
constexpr int STW_BYTES = TN * SG * 2;  // 3072: d_w fp16 [TN rows][8 blocks] (TMA box 8 x 192)
constexpr int STX_BYTES = TM * SG * 4;  // 4096: dx f32 [TM tokens][8 blocks] (TMA box 8 x 128)
constexpr int ST_BYTES = STW_BYTES + STX_BYTES;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + S * A_BYTES;
constexpr int OFF_RAW = OFF_B + S * B_BYTES;
constexpr int OFF_SCL = OFF_RAW + RAW * RB_BYTES;
constexpr int OFF_STILE = OFF_SCL + SR * SCL_BYTES;
constexpr int OFF_BAR = OFF_STILE + STG * ST_BYTES;
// afull, opempty, full per operand stage; rfull, rempty per raw stage;
// dfull, dempty per D buffer; drain; sfull, sempty per scale tile stage
constexpr int N_BARS = 3 * S + 2 * RAW + 2 * NDBUF + 1 + 2 * STG;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16;

static_assert((RAW & (RAW - 1)) == 0 && (S & (S - 1)) == 0 && (SR & (SR - 1)) == 0 && (NDBUF & (NDBUF - 1)) == 0,
              "ring sizes are powers of two");
static_assert(S == SG, "the prologue converts exactly the first scale tile's blocks");
static_assert(OFF_STILE % 128 == 0 && ST_BYTES % 128 == 0 && STW_BYTES % 128 == 0, "scale tile alignment");
static_assert(OFF_B % 1024 == 0 && OFF_RAW % 1024 == 0 && RB_BYTES % 1024 == 0 && OFF_SCL % 16 == 0 &&
                  OFF_BAR % 8 == 0 && SMEM_BYTES <= 232448,
              "shared memory layout");
static_assert(NWORK * 2 == TN * 4, "two 8-element nibble groups per worker thread");

// ---------------------------------------------------------------- activation operand chunks
// Thread p writes 16 bytes at offset 16*p of the workspace: chunk p/512 =
// (token tile T, block b) in T-major order, and inside the chunk the 8-element
// group at op_off(row, kg) = 16*(p % 512).  Tokens past M are zeros.
__global__ void __launch_bounds__(256) k_xq_to_ops(const int8_t *__restrict__ Xq, uint4 *__restrict__ Xh, int K,
                                                   int M, long long npieces)
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
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (t < M) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(Xq + t * K + b * KB + kg * 8));
            o = s8x8_to_f16(v.x, v.y);
        }
        Xh[p] = o;
    }
}

struct Work {
    int ntm, ntiles, nb;
};

// Position of one block in this CTA's sequence: tile index, K block, and the
// tile's first token and row.  Advancing never divides.
struct Cursor {
    int tile, b, t0, r0;
};
__device__ __forceinline__ void cursor_set(const Work &w, Cursor &c, int tile)
{
    c.tile = tile;
    c.b = 0;
    const int tr = tile / w.ntm;
    c.t0 = (tile - tr * w.ntm) * TM;
    c.r0 = tr * TN;
}
__device__ __forceinline__ void cursor_next(const Work &w, Cursor &c)
{
    if (++c.b == w.nb) cursor_set(w, c, c.tile + static_cast<int>(gridDim.x));
}

// Scale of the block at cursor c for worker thread i: i < TM loads dx of
// token t0+i, TM <= i < TM + TN loads d_w of row r0 + i - TM (0 past the end).
__device__ __forceinline__ float load_scale(const Work &w, const Cursor &c, int i, const uint16_t *dsc,
                                            const float *dx, int rows, int M)
{
    if (i < TM) {
        const int t = c.t0 + i;
        return (t < M && dx != nullptr) ? __ldg(dx + static_cast<size_t>(t) * w.nb + c.b) : 0.f;
    }
    if (i < TM + TN) {
        const int r = c.r0 + i - TM;
        return (r < rows) ? __half2float(__ushort_as_half(__ldg(dsc + static_cast<size_t>(r) * w.nb + c.b))) : 0.f;
    }
    return 0.f;
}

// acc[a0 + c] (+)= dx_t * d_w[col0 + c] * d[c] for the 16 columns of one
// tensor-memory load; kFirst (the tile's first block) overwrites.  The
// empty asm keeps these FMAs ahead of the next load, so only 16 loaded
// columns are live at a time.
template <bool kFirst>
__device__ __forceinline__ void fold16(float (&acc)[EPI_COLS], const float (&d)[16], const float *scl, float dxt,
                                       int col0, int a0)
{
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
        const float4 wv = *reinterpret_cast<const float4 *>(scl + TM + col0 + c);
        const float2 s01 = __fmul2_rn(make_float2(dxt, dxt), make_float2(wv.x, wv.y));
        const float2 s23 = __fmul2_rn(make_float2(dxt, dxt), make_float2(wv.z, wv.w));
        float2 a01, a23;
        if (kFirst) {
            a01 = __fmul2_rn(s01, make_float2(d[c], d[c + 1]));
            a23 = __fmul2_rn(s23, make_float2(d[c + 2], d[c + 3]));
        } else {
            a01 = __ffma2_rn(s01, make_float2(d[c], d[c + 1]), make_float2(acc[a0 + c], acc[a0 + c + 1]));
            a23 = __ffma2_rn(s23, make_float2(d[c + 2], d[c + 3]), make_float2(acc[a0 + c + 2], acc[a0 + c + 3]));
        }
        acc[a0 + c] = a01.x;
        acc[a0 + c + 1] = a01.y;
        acc[a0 + c + 2] = a23.x;
        acc[a0 + c + 3] = a23.y;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) asm volatile("" : "+f"(acc[a0 + c]));
}

// ---------------------------------------------------------------- the kernel
template <bool kDumpD>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_q8act_tc(const uint8_t *__restrict__ Xh, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX, int tiles,
                    const uint16_t *__restrict__ dsc, const float *__restrict__ dx, float *__restrict__ Y,
                    int32_t *__restrict__ Dout, int rows, int K, int M, int *__restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_afull = sbase + OFF_BAR, bar_opempty = bar_afull + 8 * S, bar_full = bar_opempty + 8 * S;
    const uint32_t bar_rfull = bar_full + 8 * S, bar_rempty = bar_rfull + 8 * RAW;
    const uint32_t bar_dfull = bar_rempty + 8 * RAW, bar_dempty = bar_dfull + 8 * NDBUF;
    const uint32_t bar_drain = bar_dempty + 8 * NDBUF;
    const uint32_t bar_sfull = bar_drain + 8, bar_sempty = bar_sfull + 8 * STG;
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
            mbar_init(bar_full + 8 * i, WORK_WARPS);
        }
        for (int i = 0; i < RAW; ++i) {
            mbar_init(bar_rfull + 8 * i, 1);
            mbar_init(bar_rempty + 8 * i, WORK_WARPS);
        }
        for (int b = 0; b < NDBUF; ++b) {
            mbar_init(bar_dfull + 8 * b, 1);
            mbar_init(bar_dempty + 8 * b, WORK_WARPS);
        }
        mbar_init(bar_drain, 1);
        for (int i = 0; i < STG; ++i) {
            mbar_init(bar_sfull + 8 * i, 1);
            mbar_init(bar_sempty + 8 * i, WORK_WARPS);
        }
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
        // ------------------------------------------------ nibble tile loads
        if (lane == 0) {
            Cursor c;
            cursor_set(w, c, static_cast<int>(blockIdx.x));
            int rs = 0;
            uint32_t rph = 0;
            int nr = 0;  // loads issued
            int gi = 0;  // scale tiles issued
            for (int gb = 0; gb < nblocks; ++gb) {
                if (tiles && (c.b & (SG - 1)) == 0) {
                    const int sg = gi & (STG - 1);
                    if (!wait_bounded(bar_sempty + 8 * sg, (static_cast<uint32_t>(gi / STG) & 1u) ^ 1u, abort, status))
                        break;
                    const uint32_t dst = sbase + OFF_STILE + sg * ST_BYTES;
                    mbar_expect_tx(bar_sfull + 8 * sg, ST_BYTES);
                    tma_load_2d(dst, &mapW, c.b, c.r0, bar_sfull + 8 * sg);
                    tma_load_2d(dst + STW_BYTES, &mapX, c.b, c.t0, bar_sfull + 8 * sg);
                    ++gi;
                }
                if (!wait_bounded(bar_rempty + 8 * rs, rph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_rfull + 8 * rs, RB_BYTES);
                tma_load_2d(sbase + OFF_RAW + rs * RB_BYTES, &mapB, c.b * 16, c.r0, bar_rfull + 8 * rs);
                ++nr;
                cursor_next(w, c);
                if (++rs == RAW) {
                    rs = 0;
                    rph ^= 1u;
                }
            }
            // No load may still be landing in shared memory when the CTA exits
            // (relevant only after an abort: normally every load has been consumed).
            volatile int no_abort = 0;
            for (int gb = (nr > RAW ? nr - RAW : 0); gb < nr; ++gb)
                wait_bounded(bar_rfull + 8 * (gb % RAW), static_cast<uint32_t>((gb / RAW) & 1), &no_abort, status);
            for (int g = (gi > STG ? gi - STG : 0); g < gi; ++g)
                wait_bounded(bar_sfull + 8 * (g % STG), static_cast<uint32_t>((g / STG) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == ACOPY_WARP) {
        // ------------------------------------------------ A operand copies
        if (lane == 0) {
            Cursor c;
            cursor_set(w, c, static_cast<int>(blockIdx.x));
            int s = 0;
            uint32_t sph = 0;
            int na = 0;  // copies issued
            for (int gb = 0; gb < nblocks; ++gb) {
                if (!wait_bounded(bar_opempty + 8 * s, sph ^ 1u, abort, status)) break;
                mbar_expect_tx(bar_afull + 8 * s, A_BYTES);
                bulk_load(sbase + OFF_A + s * A_BYTES,
                          Xh + (static_cast<size_t>(c.t0 / TM) * w.nb + c.b) * static_cast<size_t>(A_BYTES), A_BYTES,
                          bar_afull + 8 * s);
                ++na;
                cursor_next(w, c);
                if (++s == S) {
                    s = 0;
                    sph ^= 1u;
                }
            }
            volatile int no_abort = 0;
            for (int gb = (na > S ? na - S : 0); gb < na; ++gb)
                wait_bounded(bar_afull + 8 * (gb % S), static_cast<uint32_t>((gb / S) & 1), &no_abort, status);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, buf = 0;
            uint32_t sph = 0, dph = 0;
            for (int gb = 0; gb < nblocks; ++gb) {
                if (!wait_bounded(bar_afull + 8 * s, sph, abort, status)) break;
                if (!wait_bounded(bar_full + 8 * s, sph, abort, status)) break;
                if (!wait_bounded(bar_dempty + 8 * buf, dph ^ 1u, abort, status)) break;
                tc_fence_after();
                const uint32_t a0 = sbase + OFF_A + s * A_BYTES, b0 = sbase + OFF_B + s * B_BYTES;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_f16(tmem + buf * DBUF, smem_desc(a0 + ks * 256, 128, 512), smem_desc(b0 + ks * 256, 128, 512),
                            kIdesc, ks);
                mma_commit(bar_dfull + 8 * buf);
                mma_commit(bar_opempty + 8 * s);
                if (++s == S) {
                    s = 0;
                    sph ^= 1u;
                }
                if (++buf == NDBUF) {
                    buf = 0;
                    dph ^= 1u;
                }
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
        // this thread's two nibble groups: row tid/2, K groups 2*(tid%2) and +1
        const int crow = tid >> 1, chalf = tid & 1;
        const uint32_t csrc = crow * 16 + chalf * 8;
        const uint32_t cdst = op_off(crow, 2 * chalf);
        bool ok = true;
        // cursors: ce = block whose D is folded, cc = block converted (S ahead).
        // Ring stages and parities follow from the block number (all ring
        // sizes are powers of two).
        Cursor ce, cc;
        cursor_set(w, ce, static_cast<int>(blockIdx.x));
        cc = ce;
        // Scale of block g for this thread from the staged scale tile (the
        // block's position in the CTA's sequence gives its tile: every tile
        // holds whole 8-block groups); the first block of a group waits for
        // the tile to land.
        auto tile_scale = [&](int g) -> float {
            const int sg = (g / SG) & (STG - 1);
            if ((g & (SG - 1)) == 0)
                ok = ok && wait_warp(bar_sfull + 8 * sg, static_cast<uint32_t>(g / (SG * STG)) & 1u, abort, status);
            const uint8_t *t = smem + OFF_STILE + sg * ST_BYTES;
            if (tid < TM) return reinterpret_cast<const float *>(t + STW_BYTES)[tid * SG + (g & (SG - 1))];
            if (tid < TM + TN)
                return __half2float(__ushort_as_half(reinterpret_cast<const uint16_t *>(t)[(tid - TM) * SG + (g & (SG - 1))]));
            return 0.f;
        };
        // stage blocks 0..S-1 (S <= RAW: their raw stages are 0..S-1, first phase)
        for (int gb = 0; gb < S && gb < nblocks && ok; ++gb) {
            const float sv = tiles ? tile_scale(gb) : load_scale(w, cc, tid, dsc, dx, rows, M);
            if (!ok) break;
            ok = wait_warp(bar_rfull + 8 * gb, 0u, abort, status);
            if (!ok) break;
            {
                const uint2 v = *reinterpret_cast<const uint2 *>(smem + OFF_RAW + gb * RB_BYTES + csrc);
                uint8_t *dst = smem + OFF_B + gb * B_BYTES + cdst;
                *reinterpret_cast<uint4 *>(dst) = nib8_to_f16(v.x);
                *reinterpret_cast<uint4 *>(dst + 128) = nib8_to_f16(v.y);
            }
            if (tid < TM + TN) reinterpret_cast<float *>(smem + OFF_SCL + gb * SCL_BYTES)[tid] = sv;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_full + 8 * gb);
                mbar_arrive(bar_rempty + 8 * gb);
                if (tiles && (gb & (SG - 1)) == SG - 1) mbar_arrive(bar_sempty + 8 * ((gb / SG) & (STG - 1)));
            }
            cursor_next(w, cc);
        }
        float acc[EPI_COLS];  // written first by each tile's block 0
        // without scale tiles, the scale of the next block to convert is
        // loaded one iteration ahead
        float sv = (!tiles && S < nblocks) ? load_scale(w, cc, tid, dsc, dx, rows, M) : 0.f;
        for (int gb = 0; gb < nblocks && ok; ++gb) {
            const int gn = gb + S;  // block converted in this iteration
            const int buf = gb & (NDBUF - 1);
            ok = wait_warp(bar_dfull + 8 * buf, static_cast<uint32_t>(gb / NDBUF) & 1u, abort, status);
            if (!ok) break;
            tc_fence_after();
            const float *scl = reinterpret_cast<const float *>(smem + OFF_SCL + (gb & (SR - 1)) * SCL_BYTES);
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
                    const int t = ce.t0 + q * 32 + lane;
                    if (t < M) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int r = ce.r0 + c0 + part * 16 + c;
                            if (r < rows)
                                Dout[(static_cast<size_t>(t) * rows + r) * w.nb + ce.b] = __float2int_rz(d[c]);
                        }
                    }
                } else if (ce.b == 0) {
                    fold16<true>(acc, d, scl, dxt, c0 + part * 16, part * 16);
                } else {
                    fold16<false>(acc, d, scl, dxt, c0 + part * 16, part * 16);
                }
            }
            if (!kDumpD && ce.b == w.nb - 1) {
                const int t = ce.t0 + q * 32 + lane;
                if (t < M) {
                    float *yrow = Y + static_cast<size_t>(t) * rows + ce.r0 + c0;
                    const int nvalid = rows - (ce.r0 + c0);
                    const bool vec = (rows & 3) == 0;
#pragma unroll
                    for (int c = 0; c < EPI_COLS; c += 4) {
                        if (vec && c + 4 <= nvalid) {
                            *reinterpret_cast<float4 *>(yrow + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (c + e < nvalid) yrow[c + e] = acc[c + e];
                        }
                    }
                }
                // (the next tile's first block overwrites the accumulators)
            }
            cursor_next(w, ce);
            // convert the nibbles of block gb + S into the stage the MMA of block gb has finished with
            if (gn < nblocks) {
                const int rs = gn & (RAW - 1), st = gn & (S - 1);
                if (tiles) {
                    sv = tile_scale(gn);
                    if (!ok) break;
                }
                ok = wait_warp(bar_rfull + 8 * rs, static_cast<uint32_t>(gn / RAW) & 1u, abort, status);
                if (!ok) break;
                {
                    const uint2 v = *reinterpret_cast<const uint2 *>(smem + OFF_RAW + rs * RB_BYTES + csrc);
                    uint8_t *dst = smem + OFF_B + st * B_BYTES + cdst;
                    *reinterpret_cast<uint4 *>(dst) = nib8_to_f16(v.x);
                    *reinterpret_cast<uint4 *>(dst + 128) = nib8_to_f16(v.y);
                }
                if (tid < TM + TN) reinterpret_cast<float *>(smem + OFF_SCL + (gn & (SR - 1)) * SCL_BYTES)[tid] = sv;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_full + 8 * st);
                    mbar_arrive(bar_rempty + 8 * rs);
                    if (tiles && (gn & (SG - 1)) == SG - 1) mbar_arrive(bar_sempty + 8 * ((gn / SG) & (STG - 1)));
                }
                cursor_next(w, cc);
                if (!tiles && gn + 1 < nblocks) sv = load_scale(w, cc, tid, dsc, dx, rows, M);
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
size_t gemm_workspace_bytes(int K, int M)
{
    if (K < tc::KB || K % tc::KB != 0 || M < 1) return 0;
    return static_cast<size_t>((M + tc::TM - 1) / tc::TM) * static_cast<size_t>(K / tc::KB) * tc::A_BYTES;
}

static int launch_tc(bool dump, const void *W, const int8_t *Xq, const float *dx, float *Y, int32_t *D,
                     void *ws, size_t ws_bytes, int rows, int K, int M, cudaStream_t s)
{
    const int nb = K / 32;
    const size_t need = gemm_workspace_bytes(K, M);
    if (need == 0) return GQ_ERR_SHAPE;
    if (ws_bytes < need) return GQ_ERR_WORKSPACE;
    const long long ntiles_ll = static_cast<long long>((M + tc::TM - 1) / tc::TM) * ((rows + tc::TN - 1) / tc::TN);
    // per-CTA block counts are ints in the kernel
    if (ntiles_ll * nb > 0x7FFFFFFFll) return GQ_ERR_SHAPE;
    const int ntiles = static_cast<int>(ntiles_ll);
    const uint8_t *nib = static_cast<const uint8_t *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb * 16);
    CUtensorMap mapB;
    if (!make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, nib, static_cast<uint64_t>(nb) * 16,
                  static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 16, 16, tc::TN))
        return GQ_ERR_CUDA;
    // Scale tiles need 16-byte row strides in both scale arrays: nb % 8 == 0.
    CUtensorMap mapW, mapX;
    std::memset(&mapW, 0, sizeof(mapW));
    std::memset(&mapX, 0, sizeof(mapX));
    const int tiles = (!dump && nb % tc::SG == 0) ? 1 : 0;
    if (tiles) {
        if (!make_map(&mapW, CU_TENSOR_MAP_DATA_TYPE_UINT16, dsc, static_cast<uint64_t>(nb),
                      static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 2, tc::SG, tc::TN) ||
            !make_map(&mapX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, static_cast<uint64_t>(nb), static_cast<uint64_t>(M),
                      static_cast<uint64_t>(nb) * 4, tc::SG, tc::TM))
            return GQ_ERR_CUDA;
    }

    // activation codes -> f16 operand chunks
    const long long npieces = static_cast<long long>(need / 16);
    long long pgrid = (npieces + 255) / 256;
    const long long pmax = static_cast<long long>(sm_count()) * 8;
    if (pgrid > pmax) pgrid = pmax;
    int rc = status_from(launch_pdl(tc::k_xq_to_ops, dim3(static_cast<unsigned>(pgrid)), dim3(256), 0, s, Xq,
                                    static_cast<uint4 *>(ws), K, M, npieces));
    if (rc != GQ_OK) return rc;

    auto kern = dump ? tc::k_gemm_q8act_tc<true> : tc::k_gemm_q8act_tc<false>;
    const int occ = ctas_per_sm(reinterpret_cast<const void *>(kern), tc::NTHREADS, tc::SMEM_BYTES);
    if (occ <= 0) return GQ_ERR_CUDA;
    int grid = sm_count();
    if (grid > ntiles) grid = ntiles;
    return status_from(launch_pdl(kern, dim3(grid), dim3(tc::NTHREADS), static_cast<size_t>(tc::SMEM_BYTES), s,
                                  static_cast<const uint8_t *>(ws), mapB, mapW, mapX, tiles, dsc, dx, Y, D, rows, K, M,
                                  status_word()));
}

int launch_gemm_q8act_tc(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes,
                         int rows, int K, int M, cudaStream_t s)
{
    return launch_tc(false, W, Xq, dx, Y, nullptr, ws, ws_bytes, rows, K, M, s);
}

int launch_block_dots_tc(const void *W, const int8_t *Xq, int32_t *D, void *ws, size_t ws_bytes, int rows, int K,
                         int M, cudaStream_t s)
{
    return launch_tc(true, W, Xq, nullptr, nullptr, D, ws, ws_bytes, rows, K, M, s);
}

}  // namespace gq
