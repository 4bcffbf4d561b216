// gq_ring.cuh -- weight streaming for the 4-bit decode matvecs through a
// per-warp ring of shared-memory stages filled by bulk copies.
//
// Why: a decode matvec reads every weight byte once, so it is bound by HBM
// bandwidth only when enough bytes are in flight per SM (Little's law: about
// 30-40 KB per SM at GB300's bandwidth and loaded latency).  Loads into
// registers tie bytes in flight to registers; here each warp owns S stages of
// shared memory, and one `cp.async.bulk` per (row, plane) fills a stage and
// completes on the stage's mbarrier.  The warp then reads nibbles, scales and
// x from shared memory only.  Weights never depend on the previous kernel,
// so the first S stages are requested before the dependent-launch wait.
//
// Work decomposition (all static, deterministic):
//   * The grid is ncl clusters of cs CTAs.  Cluster c takes a near-equal
//     contiguous share of the rows; CTA rank r of the cluster takes the r-th
//     near-equal slice of K (in units of `unit`), so cs > 1 is a split-K for
//     short-wide shapes.  The ranks' partial row sums are added by rank 0 in
//     rank order through distributed shared memory.
//   * Inside a CTA, each of the W warps takes q whole groups of NR rows over
//     the CTA's whole K slice (phase A); the fewer than W NR rows left are
//     shared by all warps, warp w taking the w-th of W slices of the CTA's K
//     slice (phase B), and their partial sums are added in warp order.
//   * A warp is 4 groups of 8 lanes; group g owns R rows of the current NR-row
//     group, lane lp takes K units lp, lp + 8, ... of the stage's chunk.  One
//     staged x block serves the group's R rows (times the NM matrices), and
//     the four groups read the same x addresses (a shared-memory broadcast).
#pragma once

#include "gq_matvec.cuh"

namespace gq {
namespace ring {

constexpr int kLG = 8;          // lanes per row group
constexpr int kG = 32 / kLG;    // row groups per warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// Launch-time geometry (chosen by the host, identical for every CTA).
struct Plan {
    int unit;      // K-split granularity in K units (Q4_0: 8 blocks, so scale copies start 16-byte aligned)
    int cs;        // CTAs per cluster = K slices per row (1: no split)
    int ring_off;  // byte offset of the ring in dynamic shared memory (after the staged x slice)
    int red_off;   // byte offset of the per-row sums of the cluster reduction
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Makes the initialised barriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_bar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Orders this thread's earlier shared-memory reads before a later bulk copy
// that overwrites the same bytes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Streaming weights are read once: L2 evict-first.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Global -> this CTA's shared memory, completing `bytes` on the mbarrier
// (src, dst 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// A waiting warp may be suspended up to this long inside one try_wait (it
// resumes as soon as the phase completes), so waiting warps leave the issue
// slots to the warps that have data.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
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
// Bounded wait for the phase of `bar` with the given parity: false (and
// GQ_ERR_TIMEOUT in the device status word) if it does not complete within
// `limit_ns`.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, int *status, uint64_t limit_ns)
{
    if (try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u && globaltimer() - t0 > limit_ns) {
            atomicExch(status, GQ_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank)
{
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Near-equal split of n items over parts: part i gets [lo, lo + cnt).
__device__ __forceinline__ void split(int n, int parts, int i, int &lo, int &cnt)
{
    const int q = n / parts, r = n % parts;
    lo = i * q + min(i, r);
    cnt = q + (i < r ? 1 : 0);
}

// ---------------------------------------------------------------- input vectors
// The staged layout is stage_x_q4's (padded 144-byte blocks); `e0` is the
// first element of the CTA's K slice and `n` its element count.
struct InX {
    const float *__restrict__ x;
    __device__ __forceinline__ void stage(float *xs, int e0, int n) const { stage_x_q4<false>(xs, x + e0, n); }
};
struct InXSum {  // with each block's sum of x (the Q4_K min term)
    const float *__restrict__ x;
    __device__ __forceinline__ void stage(float *xs, int e0, int n) const { stage_x_q4<true>(xs, x + e0, n); }
};
// gelu_tanh(g) * u, formed in f32 while staging (the gated down projection).
struct InGeglu {
    const float *__restrict__ g;
    const float *__restrict__ u;
    __device__ __forceinline__ void stage(float *xs, int e0, int n) const
    {
        const float *gp = g + e0, *up = u + e0;
        for (int i = threadIdx.x; i < (n >> 3); i += blockDim.x) {
            const float4 g0 = *reinterpret_cast<const float4 *>(gp + 8 * i);
            const float4 g1 = *reinterpret_cast<const float4 *>(gp + 8 * i + 4);
            const float4 u0 = *reinterpret_cast<const float4 *>(up + 8 * i);
            const float4 u1 = *reinterpret_cast<const float4 *>(up + 8 * i + 4);
            const float4 a = make_float4(gelu_tanh(g0.x) * u0.x, gelu_tanh(g0.y) * u0.y, gelu_tanh(g0.z) * u0.z,
                                         gelu_tanh(g0.w) * u0.w);
            const float4 b = make_float4(gelu_tanh(g1.x) * u1.x, gelu_tanh(g1.y) * u1.y, gelu_tanh(g1.z) * u1.z,
                                         gelu_tanh(g1.w) * u1.w);
            float *dst = xs + (i >> 2) * kXBlk + 8 * (i & 3);
            *reinterpret_cast<float4 *>(dst) = make_float4(a.x, b.x, a.y, b.y);
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(a.z, b.z, a.w, b.w);
        }
        __syncthreads();
    }
};

// ---------------------------------------------------------------- formats
template <int NM>
struct Q40Src {
    const uint8_t *nib[NM];  // nibble planes
    const uint8_t *sc[NM];   // scale planes
};
struct Q4KSrc {
    const uint8_t *nib;  // nibble plane
    const uint8_t *rec;  // record plane
};

// Packed Q4_0 (one or two matrices with the same shape: the FFN's gate and
// up).  K unit = one 32-weight block.  A stage holds, per matrix, NR rows of
// KC 16-byte nibble payloads, then NR rows of KC fp16 scales padded to
// 2 KC + 16 bytes (so the four row groups' scale reads fall on distinct
// banks).  KC is a compile-time multiple of 8: every shared-memory offset of
// the consumer loop is an immediate.
template <int NM, int R, int KC>
struct Q40 {
    static_assert(KC % 8 == 0, "whole 8-block groups per chunk");
    static constexpr int kNM = NM;
    static constexpr int kNR = kG * R;
    static constexpr int kKC = KC;
    static constexpr int kXPerUnit = 1;  // staged x blocks per K unit
    static constexpr int kScStride = 2 * KC + 16;
    static constexpr int kMatBytes = kNR * (18 * KC + 16);
    static constexpr int kStageBytes = NM * kMatBytes;
    using Src = Q40Src<NM>;

    // Lane j < NM n copies nibble row (m, r); lane 16 + j its scales.
    static __device__ __forceinline__ void issue(const Src &s, uint32_t stg, uint32_t bar, int lane, int row0, int n,
                                                 int k0, int kcu, int nk, uint64_t pol)
    {
        if (lane == 0) arrive_expect_tx(bar, static_cast<uint32_t>(NM * n * kcu * 18));
        __syncwarp();
        const int j = lane & 15;
        if (j < NM * n) {
            const int m = j < n ? 0 : 1, r = j - m * n;
            const size_t blk = static_cast<size_t>(row0 + r) * nk + k0;
            const uint32_t base = stg + m * kMatBytes;
            // (a select, not an index: the source pointers stay in registers)
            const uint8_t *nib = (NM == 1 || m == 0) ? s.nib[0] : s.nib[NM - 1];
            const uint8_t *sc = (NM == 1 || m == 0) ? s.sc[0] : s.sc[NM - 1];
            if (lane < 16)
                bulk_g2s(base + r * KC * 16, nib + blk * 16, kcu * 16, bar, pol);
            else
                bulk_g2s(base + kNR * KC * 16 + r * kScStride, sc + blk * 2, kcu * 2, bar, pol);
        }
    }

    // acc[m R + i] += the dot products of group g's rows over the stage's
    // kcu (<= KC) blocks; xk = the staged x block of the chunk's first block.
    static __device__ __forceinline__ void compute(const uint8_t *stg, const float *xk, int kcu, int g, int lp,
                                                   float2 (&acc)[NM * R])
    {
        const uint8_t *wrow = stg + (g * R) * KC * 16 + lp * 16;
        const uint16_t *srow = reinterpret_cast<const uint16_t *>(stg + kNR * KC * 16 + (g * R) * kScStride) + lp;
        const float *xl = xk + lp * kXBlk;
#pragma unroll
        for (int it = 0; it < KC / kLG; ++it) {
            if (lp + it * kLG < kcu) {
                uint4 w[NM * R];
                float d[NM * R];
#pragma unroll
                for (int m = 0; m < NM; ++m)
#pragma unroll
                    for (int i = 0; i < R; ++i) {
                        w[m * R + i] = *reinterpret_cast<const uint4 *>(wrow + m * kMatBytes + i * KC * 16 +
                                                                        it * kLG * 16);
                        d[m * R + i] = half_bits_to_float(
                            *(srow + (m * kMatBytes + i * kScStride) / 2 + it * kLG));
                    }
                float2 blk[NM * R];
                q4_block<8, NM * R>(w, xl + it * kLG * kXBlk, blk);
#pragma unroll
                for (int j = 0; j < NM * R; ++j) acc[j] = ffma2(blk[j], mk2(d[j], d[j]), acc[j]);
            }
        }
    }
};

// Packed Q4_K.  K unit = one 256-weight super-block (8 sub-blocks; lane lp of
// a group always takes sub-block lp).  A stage holds NR rows of KC 128-byte
// nibble payloads, then NR rows of KC 16-byte records {d, dmin, scales}
// padded to 16 KC + 16 bytes.
template <int R, int KC>
struct Q4K {
    static constexpr int kNM = 1;
    static constexpr int kNR = kG * R;
    static constexpr int kKC = KC;
    static constexpr int kXPerUnit = 8;
    static constexpr int kRecStride = 16 * KC + 16;
    static constexpr int kStageBytes = kNR * (144 * KC + 16);
    using Src = Q4KSrc;

    static __device__ __forceinline__ void issue(const Src &s, uint32_t stg, uint32_t bar, int lane, int row0, int n,
                                                 int k0, int kcu, int nk, uint64_t pol)
    {
        if (lane == 0) arrive_expect_tx(bar, static_cast<uint32_t>(n * kcu * 144));
        __syncwarp();
        const int r = lane & 15;
        if (r < n) {
            const size_t sb = static_cast<size_t>(row0 + r) * nk + k0;
            if (lane < 16)
                bulk_g2s(stg + r * KC * 128, s.nib + sb * 128, kcu * 128, bar, pol);
            else
                bulk_g2s(stg + kNR * KC * 128 + r * kRecStride, s.rec + sb * 16, kcu * 16, bar, pol);
        }
    }

    static __device__ __forceinline__ void compute(const uint8_t *stg, const float *xk, int kcu, int g, int lp,
                                                   float2 (&acc)[R])
    {
        const Q4KSub sub = q4k_sub(lp);
        const uint8_t *wrow = stg + (g * R) * KC * 128 + lp * 16;
        const uint8_t *rrow = stg + kNR * KC * 128 + (g * R) * kRecStride;
        const float *xl = xk + lp * kXBlk;
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            if (j < kcu) {
                const float *xb = xl + 8 * j * kXBlk;
                uint4 w[R], rc[R];
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    w[i] = *reinterpret_cast<const uint4 *>(wrow + i * KC * 128 + j * 128);
                    rc[i] = *reinterpret_cast<const uint4 *>(rrow + i * kRecStride + j * 16);
                }
                float2 blk[R];
                q4_block<0, R>(w, xb, blk);
                const float xsum = xb[32];
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    float dsc, dm;
                    q4k_dm(rc[i], sub, dsc, dm);
                    acc[i] = ffma2(blk[i], mk2(dsc, dsc), acc[i]);
                    acc[i].x = fmaf(-dm, xsum, acc[i].x);
                }
            }
        }
    }
};

// ---------------------------------------------------------------- outputs
struct OutY {  // y[row] = s
    float *__restrict__ y;
    __device__ __forceinline__ void put(int row, const float (&s)[1]) const { y[row] = s[0]; }
};
struct OutGeglu {  // h[row] = gelu_tanh(gate) * up
    float *__restrict__ h;
    __device__ __forceinline__ void put(int row, const float (&s)[2]) const { h[row] = gelu_tanh(s[0]) * s[1]; }
};

// ---------------------------------------------------------------- the kernel
// One warp's stage sequence: phase A (q groups of NR rows over the CTA's K
// slice), then phase B (the left-over rows, in groups of at most NR, over the
// warp's slice of the CTA's K slice); each group's K range in chunks of <= KC.
// A cursor walks it without divisions.
struct Seq {
    int a_row0, q, a_k0, a_nch, a_kn;      // phase A
    int b_row0, nleft, b_k0, b_nch, b_kn;  // phase B
    int n;                                  // units in all
};
struct Cursor {
    int phase, grp, ch;  // phase 0: A, 1: B
};
struct Unit {
    int row0, rows, k0, kcu;
    bool first, last, phase_b;
};
template <int NR, int KC>
__device__ __forceinline__ Unit unit_at(const Seq &s, const Cursor &c)
{
    Unit u;
    u.phase_b = c.phase != 0;
    const int nch = u.phase_b ? s.b_nch : s.a_nch;
    u.row0 = (u.phase_b ? s.b_row0 : s.a_row0) + c.grp * NR;
    u.rows = u.phase_b ? min(NR, s.nleft - c.grp * NR) : NR;
    u.k0 = (u.phase_b ? s.b_k0 : s.a_k0) + c.ch * KC;
    u.kcu = min(KC, (u.phase_b ? s.b_kn : s.a_kn) - c.ch * KC);
    u.first = c.ch == 0;
    u.last = c.ch == nch - 1;
    return u;
}
__device__ __forceinline__ void advance(const Seq &s, Cursor &c)
{
    const int nch = c.phase ? s.b_nch : s.a_nch;
    if (++c.ch == nch) {
        c.ch = 0;
        if (++c.grp == s.q && c.phase == 0) {
            c.phase = 1;
            c.grp = 0;
        }
    }
}

// F: format (Q40<NM,R,KC> or Q4K<R,KC>), W: warps per CTA, S: stages per
// warp, In: input vector, Out: output mapping.  nk = K units per row.
template <class F, int R, int W, int S, class In, class Out>
__global__ void __launch_bounds__(W * 32, (W <= 8 ? 2 : 1))
    k_ring_matvec(typename F::Src src, In in, Out out, int rows, int nk, Plan p, int *status)
{
    constexpr int NM = F::kNM, NR = F::kNR, KC = F::kKC, SB = F::kStageBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[W][S];
    __shared__ float pb[W][W * NR][NM];  // phase-B partial sums [warp][row][matrix]

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / kLG, lp = lane % kLG;
    const int cs = p.cs;
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int ncl = static_cast<int>(gridDim.x) / cs, cl = static_cast<int>(blockIdx.x) / cs;

    // rows of this cluster, K slice of this CTA
    int r_lo, r_n, u_lo, u_n;
    split(rows, ncl, cl, r_lo, r_n);
    split(nk / p.unit, cs, rank, u_lo, u_n);
    const int k_lo = u_lo * p.unit, k_n = u_n * p.unit;

    Seq sq;
    sq.q = r_n / (W * NR);
    sq.a_row0 = r_lo + warp * sq.q * NR;
    sq.a_k0 = k_lo;
    sq.a_kn = k_n;
    sq.a_nch = (k_n + KC - 1) / KC;
    sq.b_row0 = r_lo + W * sq.q * NR;
    sq.nleft = r_n - W * sq.q * NR;
    {
        int s_lo, s_n;
        split(u_n, W, warp, s_lo, s_n);
        sq.b_k0 = k_lo + s_lo * p.unit;
        sq.b_kn = s_n * p.unit;
    }
    sq.b_nch = (sq.b_kn + KC - 1) / KC;
    sq.n = sq.q * sq.a_nch + ((sq.nleft + NR - 1) / NR) * sq.b_nch;

    uint8_t *ring = smem + p.ring_off + warp * S * SB;
    const uint32_t ring_s = saddr(ring);
    const uint32_t bar0 = saddr(&bars[warp][0]);
    const uint64_t pol = evict_first_policy();

    // phase-B partials start at zero (a warp with an empty K slice adds nothing)
    for (int t = lane; t < W * NR; t += 32)
#pragma unroll
        for (int m = 0; m < NM; ++m) pb[warp][t][m] = 0.f;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) bar_init(bar0 + 8 * s, 1);
        fence_bar_init();
    }
    __syncwarp();

    // Weights never depend on the previous kernel: request the first stages now.
    Cursor ic = {sq.q > 0 ? 0 : 1, 0, 0};  // issue cursor
    const Cursor start = ic;
#pragma unroll
    for (int s = 0; s < S; ++s)
        if (s < sq.n) {
            const Unit u = unit_at<NR, KC>(sq, ic);
            F::issue(src, ring_s + s * SB, bar0 + 8 * s, lane, u.row0, u.rows, u.k0, u.kcu, nk, pol);
            advance(sq, ic);
        }
    pdl_launch_dependents();
    pdl_wait();
    float *xs = reinterpret_cast<float *>(smem);
    in.stage(xs, k_lo * F::kXPerUnit * 32, k_n * F::kXPerUnit * 32);  // ends with a CTA barrier

    float *red = reinterpret_cast<float *>(smem + p.red_off);  // [row of the cluster][matrix], cs > 1
    float2 acc[NM * R];
    Cursor cc = start;  // consume cursor
    int i = 0;
    for (; i < sq.n; ++i) {
        const Unit u = unit_at<NR, KC>(sq, cc);
        const int st = i % S;
        if (!__all_sync(0xffffffffu, wait_bounded(bar0 + 8 * st, (i / S) & 1, status, kWaitLimitNs))) break;
        if (u.first) {
#pragma unroll
            for (int j = 0; j < NM * R; ++j) acc[j] = mk2(0.f, 0.f);
        }
        if (g * R < u.rows)
            F::compute(ring + st * SB, xs + (u.k0 - k_lo) * F::kXPerUnit * kXBlk, u.kcu, g, lp, acc);
        if (u.last) {
#pragma unroll
            for (int ii = 0; ii < R; ++ii) {
                float s[NM];
#pragma unroll
                for (int m = 0; m < NM; ++m) s[m] = group_sum<kLG>(acc[m * R + ii].x + acc[m * R + ii].y);
                const int rl = g * R + ii;
                if (lp == 0 && rl < u.rows) {
                    const int row = u.row0 + rl;
                    if (u.phase_b) {
#pragma unroll
                        for (int m = 0; m < NM; ++m) pb[warp][row - sq.b_row0][m] = s[m];
                    } else if (cs == 1) {
                        out.put(row, s);
                    } else {
#pragma unroll
                        for (int m = 0; m < NM; ++m) red[(row - r_lo) * NM + m] = s[m];
                    }
                }
            }
        }
        advance(sq, cc);
        __syncwarp();
        if (i + S < sq.n) {
            const Unit v = unit_at<NR, KC>(sq, ic);
            fence_proxy_async();
            __syncwarp();
            F::issue(src, ring_s + st * SB, bar0 + 8 * st, lane, v.row0, v.rows, v.k0, v.kcu, nk, pol);
            advance(sq, ic);
        }
    }
    if (i < sq.n) {
        // Timed out: give the copies still in flight a short, bounded chance to
        // land before the CTA's shared memory is released.
        for (int j = i; j < sq.n && j < i + S; ++j)
            wait_bounded(bar0 + 8 * (j % S), (j / S) & 1, status, kWaitLimitNs / 64);
    }

    __syncthreads();
    // phase B: add the W warps' partials in warp order
    for (int t = threadIdx.x; t < sq.nleft; t += W * 32) {
        float s[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) v += pb[w][t][m];
            s[m] = v;
        }
        if (cs == 1) {
            out.put(sq.b_row0 + t, s);
        } else {
#pragma unroll
            for (int m = 0; m < NM; ++m) red[(sq.b_row0 - r_lo + t) * NM + m] = s[m];
        }
    }
    if (cs > 1) {
        // split-K: rank 0 adds the ranks' row sums in rank order
        cluster_sync();
        if (rank == 0) {
            for (int t = threadIdx.x; t < r_n; t += W * 32) {
                float s[NM];
#pragma unroll
                for (int m = 0; m < NM; ++m) {
                    float v = red[t * NM + m];
                    for (int r = 1; r < cs; ++r) v += ld_cluster_f32(saddr(&red[t * NM + m]), r);
                    s[m] = v;
                }
                out.put(r_lo + t, s);
            }
        }
        cluster_sync();  // no CTA leaves while its sums may still be read
    }
}

}  // namespace ring
}  // namespace gq
