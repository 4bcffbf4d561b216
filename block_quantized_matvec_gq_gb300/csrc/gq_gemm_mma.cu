// gq_gemm_mma.cu -- the Q4_0 x Q8_0 contraction for token batches of up to
// about a hundred (passes of 32 tokens), with the exact integer block dots
// formed on the register-operand tensor-core path (mma.sync m16n8k16, f16
// operands that hold small integers, f32 accumulators).
//
// "Gemma 4 M4 Max kernel roadmap", K3 "prefill path" (batched Q4_0 kernels:
// integer block dots, then the two block scales applied in f32):
//   D[t][r][b] = sum_{j<32} Xq[t][32b+j] * (q_w[r][32b+j] - 8)   (exact)
//   Y[t][r]    = sum_b (d_w[r][b] * dx[t][b]) * D[t][r][b]       (f32)
//
// Operands.  Weights are the 16-row A operand, tokens the 8-column B
// operand.  Inside every 8-element group of a block both operands list the
// elements in the order 0,4,1,5,2,6,3,7 (the order the nibble unpacking
// produces), so each lane's A fragment of a block is one 32-bit nibble word
// of its row: lane (g, t) of a warp holds word t of rows g and g + 8, which
// `ldmatrix` delivers straight from the weight tile.  A = q - 8 and
// B = Xq are exact in f16, every product is an integer of magnitude at most
// 8 * 128, and a block's two MMAs (K = 16 each) start from zero, so the f32
// accumulator holds the exact block dot D (|D| <= 32768 < 2^24).  The fold
// Y += (d_w * dx) * D runs in packed f32x2 on the accumulators, in
// registers: there is no per-block read-out.
//
// Data flow (one CTA per SM, persistent over row groups of 16 * 3 * mg rows):
// * a pre-pass writes the activation image once per call: per (block b,
//   8-token tile) XB = 544 bytes = the 32 lanes' B fragments (16 bytes each:
//   token g = lane / 4, elements 8t .. 8t + 7 of the block, t = lane % 4, as
//   f16 in group order) and the tile's 8 dx of block b; tokens past M and
//   blocks past the last pad the image with zeros;
// * stages of KC = 16 blocks go through a ring of mbarrier stages: the weight
//   tile as two TMA boxes [rows][128 B] with the 128-byte swizzle
//   (conflict-free ldmatrix; two boxes per row back to back stream faster
//   than one), the d_w tile [rows][16 fp16] by TMA, the image chunk
//   [16 blocks][NT tiles][XB] by one bulk copy (every CTA reads the image
//   from L2).  Thread 0 issues the first stages, every weight tile before it
//   waits for the image (the pre-pass's output); afterwards the last warp to
//   finish with a stage issues its refill;
// * warps come in m-groups of four: warp (mg, q) takes the group's 3 m-tiles
//   and quarter q of every stage's blocks (12 warps at mg = 3, three per SM
//   sub-partition: one warp issues at most one mma.sync every ~9 cycles, so
//   every sub-partition needs the same share).  Per block a warp converts
//   its 6 nibble words (one lop3 per pair, one f16x2 add or fma per pair),
//   then per token tile loads the B fragment and the dx pair, issues two
//   MMAs per m-tile and folds.  The four quarters' partial sums are added in
//   the fixed order q0 + q1 + q2 + q3 through shared memory, so results are
//   reproducible bit for bit.
// Every mbarrier wait is bounded (2 s by %globaltimer); on timeout the CTA
// raises its abort flag and GQ_ERR_TIMEOUT in the device status word, every
// warp leaves its loops, and thread 0 waits (bounded) for the copies still
// in flight before the CTA exits.
#include <stdlib.h>

#include "gq_tc.cuh"

namespace gq {
namespace mmak {

using namespace tcu;

constexpr int kMaxKc = 16;              // blocks per stage: 8 or 16 (one or two 128-byte boxes per row)
constexpr int XB = 544;                 // image bytes per (block, 8-token tile)
constexpr int kMaxStages = 8;
constexpr int kMtPerGroup = 3;          // m-tiles (16 rows) per m-group
constexpr int kMaxMg = 3;               // m-groups per CTA
constexpr int kQuarters = 4;            // K quarters of a stage: 2 blocks each, one warp each
constexpr int kMaxThreads = 32 * kQuarters * kMaxMg;
constexpr int kPassTiles = 4;           // 8-token tiles per pass (32 tokens)

struct Args {
    const uint8_t *img;  // this pass's activation image
    float *Y;            // Y of this pass's first token ([m][rows], row stride `rows`)
    int rows, nb, m;     // weight rows, blocks per row, tokens in this pass
    int mg, ngroups, stages;
    int *status;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d = A(16x16, f16) * B(16x8, f16) + c, f32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4])
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// (y0, y1) += (dw * dx0, dw * dx1) * (d0, d1), each product and sum rounded
// to f32 as in the scalar (d_w * dx) * D fold.
__device__ __forceinline__ void fold2(float &y0, float &y1, float dw, float dx0, float dx1, float d0, float d1)
{
    asm("{\n .reg .b64 w, x, s, d, y;\n"
        " mov.b64 w, {%2, %2};\n mov.b64 x, {%3, %4};\n mul.rn.f32x2 s, w, x;\n"
        " mov.b64 d, {%5, %6};\n mov.b64 y, {%0, %1};\n fma.rn.f32x2 y, s, d, y;\n mov.b64 {%0, %1}, y;\n}"
        : "+f"(y0), "+f"(y1)
        : "f"(dw), "f"(dx0), "f"(dx1), "f"(d0), "f"(d1));
}

__host__ __device__ constexpr uint32_t stage_w_bytes(int mt, int kc) { return static_cast<uint32_t>(mt * 16 * kc * 16); }
__host__ __device__ constexpr uint32_t stage_d_bytes(int mt, int kc) { return static_cast<uint32_t>(mt * 16 * kc * 2); }
__host__ __device__ constexpr uint32_t stage_x_bytes(int nt, int kc) { return static_cast<uint32_t>(kc * nt * XB); }
// Stage layout: the weight tile as kc / 8 boxes [16 mt rows][128 B] (each
// 1024-byte aligned for the swizzle), the d_w tile [16 mt rows][kc fp16],
// the image chunk [kc blocks][nt tiles][XB]; stages padded to 1024 bytes.
__host__ __device__ constexpr uint32_t stage_bytes(int mt, int nt, int kc)
{
    return (stage_w_bytes(mt, kc) + stage_d_bytes(mt, kc) + stage_x_bytes(nt, kc) + 1023u) & ~1023u;
}

// Pre-pass: the activation image of every pass.  Pass p holds tiles
// [4p, 4p + 4) (its image starts at p * nb * 4 * XB); the last pass holds
// the remaining tiles rounded up to 1, 2 or 4 (zero tokens pad it).  One
// thread per (pass, block, tile, lane): 16 bytes of B fragment, and for
// t = 0 the token's dx of the block.
__host__ __device__ inline int pass_tiles(int tiles_left) { return tiles_left >= 3 ? kPassTiles : tiles_left; }

__global__ void __launch_bounds__(256) k_xq_image(const int8_t *__restrict__ Xq, const float *__restrict__ dx,
                                                  uint8_t *__restrict__ img, int K, int M, int nbp, long long nunits)
{
    pdl_launch_dependents();
    pdl_wait();
    const int nb = K / 32;  // blocks nb .. nbp - 1 pad the last stage with zeros
    const int ntiles = (M + 7) / 8;
    const long long per_pass = static_cast<long long>(nbp) * kPassTiles * 32;
    for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < nunits;
         u += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(u / per_pass);
        const long long within = u - p * per_pass;
        const int ntp = pass_tiles(ntiles - p * kPassTiles);
        const int b = static_cast<int>(within / (ntp * 32));
        const int rem = static_cast<int>(within - static_cast<long long>(b) * ntp * 32);
        const int n = rem >> 5, L = rem & 31, g = L >> 2, t = L & 3;
        const int tok = p * kPassTiles * 8 + n * 8 + g;
        uint8_t *tile = img + static_cast<size_t>(p) * per_pass / 32 * XB + (static_cast<size_t>(b) * ntp + n) * XB;
        uint4 frag = make_uint4(0u, 0u, 0u, 0u);
        float d = 0.f;
        if (tok < M && b < nb) {
            const uint2 c = __ldg(reinterpret_cast<const uint2 *>(Xq + static_cast<size_t>(tok) * K + b * 32 + t * 8));
            frag = s8x8_to_f16(c.x, c.y);
            d = __ldg(dx + static_cast<size_t>(tok) * nb + b);
        }
        reinterpret_cast<uint4 *>(tile)[L] = frag;
        if (t == 0) reinterpret_cast<float *>(tile + 512)[g] = d;
    }
}

template <int NT, int KC>
__global__ void __launch_bounds__(kMaxThreads, 1)
    k_gemm_mma(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapD, const Args a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kMaxStages], red_ready[kMaxMg], red_free[kMaxMg];
    __shared__ int abort_flag;
    __shared__ int slot_done[kMaxStages];  // warps finished with the slot's current stage
    __shared__ unsigned long long n_issued;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = kMtPerGroup * a.mg;
    const int ncons = kQuarters * a.mg;  // consumer warps (all of them)
    const int S = a.stages;
    const uint32_t SB = stage_bytes(mt, NT, KC), WB = stage_w_bytes(mt, KC), DB = stage_d_bytes(mt, KC);
    const uint32_t BOX = stage_w_bytes(mt, 8);  // one [16 mt rows][128 B] weight box
    const int nkc = (a.nb + KC - 1) / KC;
    volatile int *abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            slot_done[s] = 0;
        }
        n_issued = 0;
        for (int m = 0; m < a.mg; ++m) {
            mbar_init(smem_u32(&red_ready[m]), kQuarters - 1);
            mbar_init(smem_u32(&red_free[m]), 1);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch_dependents();

    // ------------------------------------------------ stage copies
    // Stage i of this CTA's sequence: row group blockIdx.x + (i / nkc) * gridDim.x,
    // 8-block chunk i % nkc.  Thread 0 issues the first S stages (every weight
    // tile before waiting for the image, which the previous kernel writes);
    // afterwards the last warp to finish with a stage issues its refill.
    const long long total =
        a.ngroups > static_cast<int>(blockIdx.x)
            ? (static_cast<long long>(a.ngroups - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1) * nkc
            : 0;
    const uint32_t tx = WB + DB + stage_x_bytes(NT, KC);
    auto issue_w = [&](long long i) {
        const int s = static_cast<int>(i % S);
        const int grp = static_cast<int>(blockIdx.x) + static_cast<int>(i / nkc) * static_cast<int>(gridDim.x);
        const int kc = static_cast<int>(i % nkc);
        const uint32_t st = base + static_cast<uint32_t>(s) * SB;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_expect_tx(fb, tx);
#pragma unroll
        for (int b = 0; b < KC / 8; ++b) tma_load_2d(st + b * BOX, &mapW, (kc * KC + 8 * b) * 16, grp * mt * 16, fb);
        tma_load_2d(st + WB, &mapD, kc * KC, grp * mt * 16, fb);
    };
    auto issue_x = [&](long long i) {
        const int s = static_cast<int>(i % S);
        const int kc = static_cast<int>(i % nkc);
        bulk_load(base + static_cast<uint32_t>(s) * SB + WB + DB,
                  a.img + static_cast<size_t>(kc) * stage_x_bytes(NT, KC), stage_x_bytes(NT, KC), smem_u32(&full[s]));
    };
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapD)) : "memory");
        const long long first = total < S ? total : S;
        for (long long i = 0; i < first; ++i) issue_w(i);
        pdl_wait();
        for (long long i = 0; i < first; ++i) issue_x(i);
        n_issued = first;
    }

    // ------------------------------------------------ consumers: m-group mgi, K quarter q
    pdl_wait();  // Y may have been written by the previous kernel
    const int q = warp & 3, mgi = warp >> 2;
    const int g = lane >> 2, t = lane & 3;
    // Quarter q takes blocks [q * KC / 4, (q + 1) * KC / 4) of every stage, in
    // pairs; ldmatrix matrices 0..3 of a pair = (rows 0-7, first block),
    // (rows 8-15, first), (rows 0-7, second), (rows 8-15, second).
    constexpr int QB = KC / 4;
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t lrow = static_cast<uint32_t>((lm & 1) * 8 + lr);
    const uint32_t qbox = static_cast<uint32_t>((q * QB) / 8) * BOX;
    constexpr int kSlot = kMtPerGroup * NT * 4 * 32;  // floats of one warp's partial sums
    float *red = reinterpret_cast<float *>(base_ptr + static_cast<size_t>(S) * SB) +
                 static_cast<size_t>(mgi) * (kQuarters - 1) * kSlot;
    long long it = 0;
    int gi = 0;
    for (int grp = blockIdx.x; grp < a.ngroups; grp += gridDim.x, ++gi) {
        const int row0 = grp * mt * 16;
        float Y[kMtPerGroup][NT][4];
#pragma unroll
        for (int m = 0; m < kMtPerGroup; ++m)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) Y[m][n][e] = 0.f;
        bool ok = true;
        for (int kc = 0; kc < nkc; ++kc, ++it) {
            const int s = static_cast<int>(it % S);
            if (!wait_warp(smem_u32(&full[s]), static_cast<uint32_t>((it / S) & 1), abort, a.status)) {
                ok = false;
                break;
            }
            const uint32_t st = base + static_cast<uint32_t>(s) * SB;
            const uint8_t *dt = base_ptr + static_cast<size_t>(s) * SB + WB;
            const uint8_t *xs = dt + DB;
#pragma unroll
            for (int bp = 0; bp < QB / 2; ++bp) {
                const int b0 = q * QB + 2 * bp;  // first block of the pair inside the stage
                const uint32_t lswz = static_cast<uint32_t>((((b0 & 7) + (lm >> 1)) ^ lr) << 4);
                uint32_t w[kMtPerGroup][4];
                uint32_t dwp[kMtPerGroup][2];  // [m-tile][row g, g + 8]: fp16 d_w of blocks b0, b0 + 1
#pragma unroll
                for (int m = 0; m < kMtPerGroup; ++m) {
                    const int jj = kMtPerGroup * mgi + m;
                    ldsm_x4(st + qbox + static_cast<uint32_t>(jj * 16 + lrow) * 128u + lswz, w[m][0], w[m][1], w[m][2],
                            w[m][3]);
                    dwp[m][0] = *reinterpret_cast<const uint32_t *>(dt + (jj * 16 + g) * (2 * KC) + 2 * b0);
                    dwp[m][1] = *reinterpret_cast<const uint32_t *>(dt + (jj * 16 + g + 8) * (2 * KC) + 2 * b0);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int blk = b0 + i;
                    uint4 A[kMtPerGroup][2];  // [m-tile][row g, row g + 8]
                    float dw[kMtPerGroup][2];
#pragma unroll
                    for (int m = 0; m < kMtPerGroup; ++m) {
                        A[m][0] = nib8_to_f16(w[m][2 * i]);
                        A[m][1] = nib8_to_f16(w[m][2 * i + 1]);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            dw[m][h] = __half2float(__ushort_as_half(
                                static_cast<unsigned short>(i == 0 ? (dwp[m][h] & 0xFFFFu) : (dwp[m][h] >> 16))));
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint8_t *tile = xs + (blk * NT + n) * XB;
                        const uint4 xb = *reinterpret_cast<const uint4 *>(tile + lane * 16);
                        const float2 dx = *reinterpret_cast<const float2 *>(tile + 512 + t * 8);
#pragma unroll
                        for (int m = 0; m < kMtPerGroup; ++m) {
                            const float z[4] = {0.f, 0.f, 0.f, 0.f};
                            float d[4];
                            mma16816(d, A[m][0].x, A[m][1].x, A[m][0].y, A[m][1].y, xb.x, xb.y, z);
                            mma16816(d, A[m][0].z, A[m][1].z, A[m][0].w, A[m][1].w, xb.z, xb.w, d);
                            fold2(Y[m][n][0], Y[m][n][1], dw[m][0], dx.x, dx.y, d[0], d[1]);
                            fold2(Y[m][n][2], Y[m][n][3], dw[m][1], dx.x, dx.y, d[2], d[3]);
                        }
                    }
                }
            }
            // The last of the CTA's warps to finish with this stage refills its buffer.
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&slot_done[s], 1) == ncons - 1) {
                    __threadfence_block();
                    slot_done[s] = 0;
                    if (it + S < total) {
                        issue_w(it + S);
                        issue_x(it + S);
                        atomicAdd(&n_issued, 1ull);
                    }
                }
            }
        }
        if (!ok) break;
        // ---- the four K quarters of the m-group, added in the fixed order q0 + q1 + q2 + q3
        const uint32_t ph = static_cast<uint32_t>(gi & 1);
        if (q != 0) {
            if (!wait_warp(smem_u32(&red_free[mgi]), ph ^ 1u, abort, a.status)) break;
            float *slot = red + (q - 1) * kSlot;
#pragma unroll
            for (int m = 0; m < kMtPerGroup; ++m)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) slot[((m * NT + n) * 4 + e) * 32 + lane] = Y[m][n][e];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&red_ready[mgi]));
            continue;
        }
        if (!wait_warp(smem_u32(&red_ready[mgi]), ph, abort, a.status)) break;
#pragma unroll
        for (int k = 0; k < kQuarters - 1; ++k)
#pragma unroll
            for (int m = 0; m < kMtPerGroup; ++m)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) Y[m][n][e] += red[k * kSlot + ((m * NT + n) * 4 + e) * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&red_free[mgi]));
        // lane (g, t) holds rows g, g + 8 x tokens 2t, 2t + 1 of each (m-tile, token tile)
#pragma unroll
        for (int m = 0; m < kMtPerGroup; ++m) {
            const int r = row0 + (kMtPerGroup * mgi + m) * 16 + g;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int tok = n * 8 + 2 * t;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = r + ((e >> 1) << 3), tt = tok + (e & 1);
                    if (rr < a.rows && tt < a.m) a.Y[static_cast<size_t>(tt) * a.rows + rr] = Y[m][n][e];
                }
            }
        }
    }
    // No copy may still be landing in shared memory when the CTA exits (only
    // possible after an abort: normally every issued stage has been consumed).
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int no_abort = 0;
        const long long n = static_cast<long long>(n_issued);
        for (long long g = (n > S ? n - S : 0); g < n; ++g)
            wait_bounded(smem_u32(&full[g % S]), static_cast<uint32_t>((g / S) & 1), &no_abort, a.status);
    }
}

}  // namespace mmak

// ---------------------------------------------------------------- host side
static int mma_passes(int M) { return ((M + 7) / 8 + mmak::kPassTiles - 1) / mmak::kPassTiles; }
static int mma_last_tiles(int M) { return mmak::pass_tiles((M + 7) / 8 - (mma_passes(M) - 1) * mmak::kPassTiles); }
static size_t mma_image_tiles(int M)
{
    return static_cast<size_t>(mma_passes(M) - 1) * mmak::kPassTiles + mma_last_tiles(M);
}
// Blocks per stage, 8 or 16.  Measured on 21504 x 5376 weights: 16 (two
// 128-byte boxes per row back to back) 23.1 / 35.9 / 103 us at M = 8 / 32 /
// 96, against 29.1 / 41.0 / 120 us with 8.
static int mma_kc(int M)
{
#ifdef GQ_TUNING
    if (const char *v = getenv("GQ_MMA_KC")) return atoi(v) == 8 ? 8 : 16;
#endif
    (void)M;
    return 16;
}

bool gemm_mma_supported(int K, int M) { return M >= 1 && K >= 256 && K % 256 == 0; }

size_t gemm_mma_workspace_bytes(int K, int M)
{
    if (!gemm_mma_supported(K, M)) return 0;
    const size_t nbp = static_cast<size_t>((K / 32 + mmak::kMaxKc - 1) / mmak::kMaxKc) * mmak::kMaxKc;
    return mma_image_tiles(M) * nbp * mmak::XB;
}

template <int NT, int KC>
static int launch_pass(const CUtensorMap &mapW, const CUtensorMap &mapD, const mmak::Args &a0, int ngroups,
                       cudaStream_t s)
{
    using namespace mmak;
    Args a = a0;
    const int mt = kMtPerGroup * a.mg;
    const uint32_t sb = stage_bytes(mt, NT, KC);
    // partial sums of K quarters 1..3 of every m-group
    const uint32_t red = static_cast<uint32_t>(a.mg * (kQuarters - 1) * kMtPerGroup * NT * 4 * 32 * 4);
    int stages = static_cast<int>((210u * 1024u - 1024u - red) / sb);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return GQ_ERR_SHAPE;
    a.stages = stages;
    const size_t smem = 1024 + static_cast<size_t>(stages) * sb + red;
    const int threads = 32 * kQuarters * a.mg;
    const int occ = ctas_per_sm(reinterpret_cast<const void *>(k_gemm_mma<NT, KC>), threads, smem);
    if (occ <= 0) return GQ_ERR_CUDA;
    int grid = sm_count() * occ;
    if (grid > ngroups) grid = ngroups;
    return status_from(launch_pdl(k_gemm_mma<NT, KC>, dim3(grid), dim3(threads), smem, s, mapW, mapD, a));
}

int launch_gemm_mma(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes, int rows,
                    int K, int M, cudaStream_t s)
{
    using namespace mmak;
    if (!gemm_mma_supported(K, M) || rows < 1) return GQ_ERR_SHAPE;
    if (ws_bytes < gemm_mma_workspace_bytes(K, M)) return GQ_ERR_WORKSPACE;
    const int nb = K / 32;
    const int kc = mma_kc(M);
    const int nbp = (nb + kc - 1) / kc * kc;
    const int nsm = sm_count();
    // m-groups of 3 m-tiles per CTA: enough that one row group per SM covers
    // the rows (21504 rows: 9 m-tiles, 150 CTAs), at most 3
    const int mtiles = (rows + 15) / 16;
    const int per_sm = (mtiles + nsm - 1) / nsm;
    int mg = (per_sm + kMtPerGroup - 1) / kMtPerGroup;
    if (mg > kMaxMg) mg = kMaxMg;
    const int mt = kMtPerGroup * mg;
    const int ngroups = (mtiles + mt - 1) / mt;
    const uint8_t *nib = static_cast<const uint8_t *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(nib + static_cast<size_t>(rows) * nb * 16);
    CUtensorMap mapW, mapD;
    if (!make_map(&mapW, CU_TENSOR_MAP_DATA_TYPE_UINT8, nib, static_cast<uint64_t>(nb) * 16,
                  static_cast<uint64_t>(rows), static_cast<uint64_t>(nb) * 16, 128, 16 * mt,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mapD, CU_TENSOR_MAP_DATA_TYPE_UINT16, dsc, static_cast<uint64_t>(nb), static_cast<uint64_t>(rows),
                  static_cast<uint64_t>(nb) * 2, static_cast<uint32_t>(kc), 16 * mt))
        return GQ_ERR_CUDA;

    // activation codes and scales -> the image of every pass
    const long long nunits = static_cast<long long>(mma_image_tiles(M)) * nbp * 32;
    long long pgrid = (nunits + 255) / 256;
    if (pgrid > static_cast<long long>(nsm) * 8) pgrid = static_cast<long long>(nsm) * 8;
    int rc = status_from(launch_pdl(k_xq_image, dim3(static_cast<unsigned>(pgrid)), dim3(256), 0, s, Xq, dx,
                                    static_cast<uint8_t *>(ws), K, M, nbp, nunits));
    if (rc != GQ_OK) return rc;

    const int np = mma_passes(M);
    for (int p = 0; p < np; ++p) {
        const int ntp = p + 1 < np ? kPassTiles : mma_last_tiles(M);
        const int tok0 = p * kPassTiles * 8;
        Args a;
        a.img = static_cast<const uint8_t *>(ws) + static_cast<size_t>(p) * nbp * kPassTiles * XB;
        a.Y = Y + static_cast<size_t>(tok0) * rows;
        a.rows = rows;
        a.nb = nb;
        a.m = M - tok0 < kPassTiles * 8 ? M - tok0 : kPassTiles * 8;
        a.mg = mg;
        a.ngroups = ngroups;
        a.stages = 0;
        a.status = status_word();
        if (kc == 16)
            rc = ntp == 1 ? launch_pass<1, 16>(mapW, mapD, a, ngroups, s)
                 : ntp == 2 ? launch_pass<2, 16>(mapW, mapD, a, ngroups, s)
                            : launch_pass<4, 16>(mapW, mapD, a, ngroups, s);
        else
            rc = ntp == 1 ? launch_pass<1, 8>(mapW, mapD, a, ngroups, s)
                 : ntp == 2 ? launch_pass<2, 8>(mapW, mapD, a, ngroups, s)
                            : launch_pass<4, 8>(mapW, mapD, a, ngroups, s);
        if (rc != GQ_OK) return rc;
    }
    return GQ_OK;
}

}  // namespace gq
