// gq_norm.cu -- RMS normalization fused with the Q8_0 quantization of the
// normalized activations, one CTA per token.
//
// "Metal kernel capability table (Phase B ground truth)", section 6:
// rms_norm scales a row by 1 / RMS and by (w + offset); rms_norm_q8 fuses
// the Q8 quantization of the normalized row into the same kernel (there the
// block scales came out wrong unless the threadgroup size and the row
// length were multiples of 32; here K % 32 == 0 is required and every
// 32-block is one group of eight lanes, as in the quantizer).
//
// The codes are integers decided by floating point, so the statistic is
// made a function of the inputs alone, independent of any summation order:
//   ss  = sum_j x_j^2, rounded once to double
//   r   = sqrt(ss / K + eps), each double operation rounded to nearest
//   inv = f32(1 / r)
//   y_j = f32(f32(x_j * inv) * f32(w_j + offset))
// followed by the Q8_0 rule of gq_quantize_q8_0 on each 32-block of y.
//
// Exact sum of squares: x = m 2^(e - 150) with m the 24-bit significand
// (e the biased exponent; subnormals take e = 1 and no hidden bit), so
// x^2 = m^2 2^(2e - 300) with m^2 < 2^48.
//
// Fast path (every row but a vanishing fraction): with E the row's largest
// exponent, each square is added to a 128-bit integer in units of
// 2^(2E - 364) (m^2 shifted left by 2(e - E) + 64, i.e. 64 bits below the
// largest square's last bit); bits shifted out below the unit are dropped,
// and a sticky flag records whether any was nonzero.  The sum A is below
// K 2^112 < 2^128, and its leading bit is at least bit 64, so the double's
// rounding position lies at least 11 bits above the unit.  The dropped part
// delta is below K units (one per term at most), so the rounding of the
// exact sum is decided by A alone unless the bits of A below the rounding
// position are within K units under the half-way point (then delta could
// carry the remainder over it): exactly half-way, the sticky flag breaks the
// tie; in the window below half-way, the row takes the slow path.
//
// Slow path: squares with the same e add exactly in a 64-bit integer bucket
// (K <= 49152 < 2^16 terms), in any order (per warp, then across the
// warps); the buckets then add exactly as B_e << 2(e - 1) into a 608-bit
// integer, which is rounded once, to nearest even, into the double
// ss = N 2^-298.
#include "gq_host.h"
#include "gq_internal.cuh"
#include "gq_q8code.cuh"

namespace gq {
namespace norm {

constexpr int kThreads = 256;
constexpr int kLimbs = 19;  // 32-bit limbs; the largest sum needs 571 bits

constexpr int kWarps = kThreads / 32;

// The squares of one element per lane into this warp's exponent buckets wb
// (non-finite values only set a flag: bit 0 for an infinity, bit 1 for a
// NaN).  Lanes with the same exponent are summed first -- the 48-bit squares
// as two 24-bit halves, whose sums over 32 lanes fit 32 bits, by full-warp
// reductions -- and lane 0 adds each exponent's sum to its bucket, so every
// bucket update is one thread's read-modify-write (no atomics, no
// same-address conflicts).
__device__ __forceinline__ void add_squares_warp(unsigned long long *wb, int *nonfinite, float f, int lane)
{
    const uint32_t b = __float_as_uint(f) & 0x7FFFFFFFu;
    uint32_t e = b >> 23, m = b & 0x7FFFFFu;
    if (e == 255u) {
        atomicOr(nonfinite, m ? 2 : 1);
        m = 0u;
    } else if (e == 0u) {
        e = 1u;  // subnormal: m 2^(1 - 150); a zero adds nothing
    } else {
        m |= 0x800000u;
    }
    const unsigned long long v = static_cast<unsigned long long>(m) * m;
    const uint32_t lo = static_cast<uint32_t>(v) & 0xFFFFFFu, hi = static_cast<uint32_t>(v >> 24);
    // one exponent per round, the lowest pending lane's; every lane leaves
    // the loop together (pending is warp-uniform and loses a bit each round)
    for (uint32_t pending = __ballot_sync(0xffffffffu, v != 0ull); pending != 0u;) {
        const uint32_t key = __shfl_sync(0xffffffffu, e, __ffs(pending) - 1);
        const bool mine = ((pending >> lane) & 1u) != 0u && e == key;
        const uint32_t slo = __reduce_add_sync(0xffffffffu, mine ? lo : 0u);
        const uint32_t shi = __reduce_add_sync(0xffffffffu, mine ? hi : 0u);
        if (lane == 0) wb[key] += (static_cast<unsigned long long>(shi) << 24) + slo;
        pending &= ~__ballot_sync(0xffffffffu, mine);
    }
}

// sum_e bucket[e] 2^(2e - 300), rounded to nearest even (one thread); occ
// marks the nonzero buckets (bit e % 32 of occ[e / 32]).
__device__ double exact_sum(const unsigned long long *bucket, const uint32_t (&occ)[8])
{
    uint32_t n[kLimbs];
    for (int i = 0; i < kLimbs; ++i) n[i] = 0u;
    for (int wd = 0; wd < 8; ++wd) {
        for (uint32_t bits = occ[wd]; bits != 0u; bits &= bits - 1u) {
            const int e = 32 * wd + __ffs(bits) - 1;
            const unsigned long long B = bucket[e];
            const int s = 2 * (e - 1), l = s >> 5, o = s & 31;  // B << s spans limbs l .. l + 2
            const unsigned long long lo = B << o;
            const uint32_t p[3] = {static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                                   o ? static_cast<uint32_t>(B >> (64 - o)) : 0u};
            unsigned long long c = 0ull;
            for (int k = 0; k < 3; ++k) {
                c += static_cast<unsigned long long>(n[l + k]) + p[k];
                n[l + k] = static_cast<uint32_t>(c);
                c >>= 32;
            }
            for (int k = l + 3; c != 0ull && k < kLimbs; ++k) {
                c += n[k];
                n[k] = static_cast<uint32_t>(c);
                c >>= 32;
            }
        }
    }
    int top = kLimbs - 1;
    while (top >= 0 && n[top] == 0u) --top;
    if (top < 0) return 0.0;
    // the 64 bits from the leading one down, and whether anything below is set
    const uint32_t a = n[top];
    const uint32_t b1 = top >= 1 ? n[top - 1] : 0u;
    const uint32_t b2 = top >= 2 ? n[top - 2] : 0u;
    bool sticky = false;
    for (int k = 0; k < top - 2; ++k) sticky |= n[k] != 0u;
    const int lz = __clz(a);
    unsigned long long v = (static_cast<unsigned long long>(a) << 32) | b1;
    if (lz) {
        v = (v << lz) | (b2 >> (32 - lz));
        sticky |= static_cast<uint32_t>(b2 << lz) != 0u;
    } else {
        sticky |= b2 != 0u;
    }
    unsigned long long m = v >> 11;  // 53 bits, leading one at bit 52
    const bool half = ((v >> 10) & 1ull) != 0ull;
    sticky |= (v & 0x3FFull) != 0ull;
    int pos = 32 * top + 31 - lz;  // bit index of the leading one of N
    if (half && (sticky || (m & 1ull))) {
        ++m;
        if (m >> 53) {  // rounded up to the next power of two
            m >>= 1;
            ++pos;
        }
    }
    // ss = m 2^(pos - 52) 2^-298: biased exponent pos - 298 + 1023, always normal
    const long long be = static_cast<long long>(pos) - 298 + 1023;
    return __longlong_as_double((be << 52) | static_cast<long long>(m & 0xFFFFFFFFFFFFFull));
}

// 64-bit shifts whose amount may reach 64: PTX clamps the amount to the
// register width, so a shift by 64 or more gives 0 (no branch needed).
__device__ __forceinline__ unsigned long long shl64(unsigned long long a, uint32_t n)
{
    unsigned long long r;
    asm("shl.b64 %0, %1, %2;" : "=l"(r) : "l"(a), "r"(n));
    return r;
}
__device__ __forceinline__ unsigned long long shr64(unsigned long long a, uint32_t n)
{
    unsigned long long r;
    asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"(a), "r"(n));
    return r;
}

// (hi, lo) += m^2 2^(2(e - E) + 64), dropping (and flagging in `sticky`)
// the bits below the unit.  Branch-free: lanes whose values differ in
// exponent take the same instructions.
__device__ __forceinline__ void add_square_fixed(uint32_t e, uint32_t m, uint32_t E, unsigned long long &lo,
                                                 unsigned long long &hi, bool &sticky)
{
    const unsigned long long sq = static_cast<unsigned long long>(m) * m;
    const int s = 2 * (static_cast<int>(e) - static_cast<int>(E)) + 64;  // <= 64
    const uint32_t sp = s > 0 ? static_cast<uint32_t>(s) : 0u;          // left shift (s >= 0)
    const uint32_t sn = s < 0 ? static_cast<uint32_t>(-s) : 0u;         // right shift (s < 0)
    const unsigned long long tl = s >= 0 ? shl64(sq, sp) : shr64(sq, sn);
    const unsigned long long th = shr64(sq, 64u - sp);  // bits at 64 and above (0 unless s > 16)
    // bits shifted out below the unit: the low min(sn, 64) bits of sq
    sticky |= s < 0 && shl64(sq, 64u - min(sn, 64u)) != 0ull;
    lo += tl;
    hi += th + (lo < tl ? 1ull : 0ull);
}

// The term of a nonzero finite x below the fast path's range (e < E - 24,
// subnormals counted as e = 1), out of line so the unrolled loops stay small:
// m^2 2^(2(e - E) + 64) < 2^48 2^16, so the term is below 2^64 units; .y is
// nonzero if bits below the unit were dropped.
__device__ __noinline__ ulonglong2 small_square(uint32_t b, uint32_t E)
{
    const uint32_t e = b >> 23;
    unsigned long long lo = 0ull, hi = 0ull;
    bool sticky = false;
    add_square_fixed(e ? e : 1u, e ? ((b & 0x7FFFFFu) | 0x800000u) : b, E, lo, hi, sticky);
    return make_ulonglong2(lo, sticky ? 1ull : 0ull);
}

// Fixed-point partial of one thread: the 128-bit sum as four 32-bit limbs
// (fast path) plus a (lo, hi, sticky) part for the rare small elements.
struct FixedAcc {
    uint32_t a0 = 0u, a1 = 0u, a2 = 0u, a3 = 0u;
    unsigned long long lo = 0ull, hi = 0ull;
    bool sticky = false;
};

// Adds x^2 for x with magnitude bits b (finite) in units of 2^(2E - 364).
// Fast path, for x with e >= E - 24 (subnormals counted as e = 1 with no
// hidden bit): with t = m << 8 (32 bits), the
// term m^2 2^(2(e - E) + 64) is t^2 2^(2k), k = e - E + 24 in [0, 24]: one
// 32 x 32 -> 64 multiply shifted by 2k < 64 into the limbs (funnel shifts
// and a one-limb select), nothing dropped.  Smaller nonzero x take small_square
// (add_square_fixed out of line).
__device__ __forceinline__ void add_square(uint32_t b, uint32_t E, FixedAcc &acc)
{
    const uint32_t e = b >> 23;
    const int k = static_cast<int>(e ? e : 1u) - static_cast<int>(E) + 24;  // subnormals: e = 1, no hidden bit
    if (k >= 0) {
        const uint32_t t = (e ? ((b & 0x7FFFFFu) | 0x800000u) : b) << 8;
        const unsigned long long p = static_cast<unsigned long long>(t) * t;
        const uint32_t p0 = static_cast<uint32_t>(p), p1 = static_cast<uint32_t>(p >> 32);
        const uint32_t k2 = 2u * static_cast<uint32_t>(k), r = k2 & 31u;
        const uint32_t l0 = p0 << r, l1 = __funnelshift_l(p0, p1, r), l2 = __funnelshift_l(p1, 0u, r);
        const bool up = k2 >= 32u;  // one limb higher
        const uint32_t c0 = up ? 0u : l0, c1 = up ? l0 : l1, c2 = up ? l1 : l2, c3 = up ? l2 : 0u;
        asm("add.cc.u32 %0, %0, %4;\n\t"
            "addc.cc.u32 %1, %1, %5;\n\t"
            "addc.cc.u32 %2, %2, %6;\n\t"
            "addc.u32 %3, %3, %7;"
            : "+r"(acc.a0), "+r"(acc.a1), "+r"(acc.a2), "+r"(acc.a3)
            : "r"(c0), "r"(c1), "r"(c2), "r"(c3));
    } else if (b != 0u) {
        const ulonglong2 t = small_square(b, E);
        acc.lo += t.x;
        acc.hi += acc.lo < t.x ? 1ull : 0ull;
        acc.sticky |= t.y != 0ull;
    }
}

// The thread's partial as (lo, hi): limbs plus the small-element part.
__device__ __forceinline__ void fixed_total(const FixedAcc &acc, unsigned long long &lo, unsigned long long &hi)
{
    const unsigned long long flo = (static_cast<unsigned long long>(acc.a1) << 32) | acc.a0;
    const unsigned long long fhi = (static_cast<unsigned long long>(acc.a3) << 32) | acc.a2;
    lo = flo + acc.lo;
    hi = fhi + acc.hi + (lo < flo ? 1ull : 0ull);
}

// The double nearest A 2^(2E - 364) given the dropped part's sticky flag,
// or a negative value if the rounding is not decided by A (K terms: the
// dropped part is below K units).
__device__ __forceinline__ double round_fixed(unsigned long long lo, unsigned long long hi, uint32_t E, bool sticky,
                                              int K)
{
    // leading bit p of A (A >= 2^64 whenever any x is nonzero; A == 0 otherwise)
    if (hi == 0ull && lo == 0ull) return sticky ? -1.0 : 0.0;
    const int p = hi ? 64 + 63 - __clzll(static_cast<long long>(hi)) : 63 - __clzll(static_cast<long long>(lo));
    if (p < 53) return -1.0;  // cannot happen for a nonzero row; take the slow path
    const int sh = p - 52;    // bits below the double's last bit
    // mantissa m53 = A >> sh, remainder r = A mod 2^sh (sh <= 75)
    unsigned long long m53, rhi, rlo;  // remainder as a 128-bit (rhi, rlo)
    if (sh >= 64) {
        m53 = hi >> (sh - 64);
        rlo = lo;
        rhi = (sh == 64) ? 0ull : (hi & ((1ull << (sh - 64)) - 1ull));
    } else {
        m53 = (lo >> sh) | (hi << (64 - sh));
        rlo = lo & ((1ull << sh) - 1ull);
        rhi = 0ull;
    }
    // half = 2^(sh - 1) as (hhi, hlo)
    const int hb = sh - 1;
    const unsigned long long hhi = hb >= 64 ? (1ull << (hb - 64)) : 0ull;
    const unsigned long long hlo = hb >= 64 ? 0ull : (1ull << hb);
    const bool r_gt = rhi > hhi || (rhi == hhi && rlo > hlo);
    const bool r_eq = rhi == hhi && rlo == hlo;
    bool up;
    if (r_gt) {
        up = true;
    } else if (r_eq) {
        up = sticky || (m53 & 1ull);
    } else {
        // below half: decided unless half - r <= K units (the dropped part could reach it)
        const unsigned long long dlo = hlo - rlo;
        const unsigned long long dhi = hhi - rhi - (hlo < rlo ? 1ull : 0ull);
        if (dhi == 0ull && dlo <= static_cast<unsigned long long>(K)) return -1.0;
        up = false;
    }
    int pos = p;
    if (up) {
        ++m53;
        if (m53 >> 53) {
            m53 >>= 1;
            ++pos;
        }
    }
    const long long be = static_cast<long long>(pos) + 2 * static_cast<long long>(E) - 364 + 1023;
    return __longlong_as_double((be << 52) | static_cast<long long>(m53 & 0xFFFFFFFFFFFFFull));
}

// Shared memory of the sum of squares of one row.
struct SumSqSmem {
    unsigned long long wbk[kWarps][256];  // per-warp exponent buckets (slow path)
    unsigned long long bucket[256];
    unsigned long long part_lo[kWarps], part_hi[kWarps];
    uint32_t emax[kWarps];
    int nonfinite;
    int slow;
    double ss;
    float inv;
};

// Block-wide: from every thread's largest magnitude bit pattern (|x| bits,
// whose unsigned order is that of the magnitudes, infinities and NaNs above
// every number), the row's largest exponent E (at least 1) returned to every
// thread, and the non-finite flags (bit 0 an infinity, bit 1 a NaN: a NaN's
// pattern is above the infinity's) set in sm.nonfinite.
__device__ __forceinline__ uint32_t block_emax(uint32_t mbits, SumSqSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    mbits = __reduce_max_sync(0xffffffffu, mbits);
    if (lane == 0) sm.emax[warp] = mbits;
    __syncthreads();
    uint32_t M = sm.emax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = max(M, sm.emax[w]);
    if (threadIdx.x == 0) sm.nonfinite = M > 0x7F800000u ? 2 : (M == 0x7F800000u ? 1 : 0);
    return max(M >> 23, 1u);
}

// Block-wide: ss from every thread's fixed-point partial (lo, hi, sticky)
// anchored at E; rows whose rounding the partials do not decide take the
// exact exponent buckets over the row in global memory.  Every thread gets
// the result.
__device__ double block_sum_squares(unsigned long long lo, unsigned long long hi, bool sticky, uint32_t E,
                                    const float4 *__restrict__ xr, int K, SumSqSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nq = K >> 2;
    // every warp adds its lanes' partials, then warp 0 the warps' sums
    // (exactly: the total stays below 2^128)
    auto add128 = [](unsigned long long &a, unsigned long long &b, unsigned long long oa, unsigned long long ob) {
        a += oa;
        b += ob + (a < oa ? 1ull : 0ull);
    };
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        add128(lo, hi, __shfl_xor_sync(0xffffffffu, lo, o), __shfl_xor_sync(0xffffffffu, hi, o));
    if (lane == 0) {
        sm.part_lo[warp] = lo;
        sm.part_hi[warp] = hi;
    }
    const int any_sticky = __syncthreads_or(sticky ? 1 : 0);
    if (threadIdx.x < 32) {
        unsigned long long a = lane < kWarps ? sm.part_lo[lane] : 0ull, b = lane < kWarps ? sm.part_hi[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            add128(a, b, __shfl_xor_sync(0xffffffffu, a, o), __shfl_xor_sync(0xffffffffu, b, o));
        if (threadIdx.x == 0) {
            double ss;
            if (sm.nonfinite & 2)
                ss = __longlong_as_double(0x7FF8000000000000ll);  // NaN
            else if (sm.nonfinite & 1)
                ss = __longlong_as_double(0x7FF0000000000000ll);  // +infinity
            else
                ss = round_fixed(a, b, E, any_sticky != 0, K);
            sm.slow = ss < 0.0 ? 1 : 0;
            sm.ss = ss;
        }
    }
    __syncthreads();
    if (sm.slow) {
        // the rounding is not decided by the fixed-point sum: exact exponent buckets
        for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) (&sm.wbk[0][0])[i] = 0ull;
        __syncthreads();
        // warp-uniform loop (the reductions use the full warp); lanes past the
        // row contribute zeros
        for (int i0 = warp * 32; i0 < nq; i0 += kThreads) {
            const int i = i0 + lane;
            const float4 v = i < nq ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            add_squares_warp(sm.wbk[warp], &sm.nonfinite, v.x, lane);
            add_squares_warp(sm.wbk[warp], &sm.nonfinite, v.y, lane);
            add_squares_warp(sm.wbk[warp], &sm.nonfinite, v.z, lane);
            add_squares_warp(sm.wbk[warp], &sm.nonfinite, v.w, lane);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < 256; e += kThreads) {  // the warps' buckets, added exactly (each total
            unsigned long long sb = 0ull;                     // stays below K 2^48 < 2^64)
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sb += sm.wbk[w][e];
            sm.bucket[e] = sb;
        }
        __syncthreads();
        if (threadIdx.x < 32) {  // warp 0: which buckets are occupied, then lane 0 adds them
            uint32_t occ[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                occ[k] = __ballot_sync(0xffffffffu, sm.bucket[32 * k + threadIdx.x] != 0ull);
            if (threadIdx.x == 0) sm.ss = exact_sum(sm.bucket, occ);
        }
        __syncthreads();
    }
    return sm.ss;
}

// The four squares of v into the fixed-point partial (a non-finite value
// adds nothing: the row's result is then decided by sm.nonfinite).
__device__ __forceinline__ void add_chunk_fixed(const float4 &v, uint32_t E, FixedAcc &acc)
{
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t b = __float_as_uint(f[k]) & 0x7FFFFFFFu;
        add_square(b < 0x7F800000u ? b : 0u, E, acc);
    }
}
// Largest magnitude bit pattern of the chunk, into mbits.
__device__ __forceinline__ void max_chunk_bits(const float4 &v, uint32_t &mbits)
{
    mbits = max(mbits, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                           max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
}

// Rows of at most kRegChunks * kThreads float4 (K <= 16384) are read once:
// thread t keeps chunks t, t + kThreads, ... in registers.
constexpr int kRegChunks = 8;

// The sum of the squares of row xr (K floats) rounded once to double
// (+infinity if the row holds an infinity, NaN if it holds a NaN); every
// thread of the CTA calls it and gets the result.  Reads the row from
// global memory (twice; a third time on the slow path).
__device__ double row_sum_squares(const float4 *__restrict__ xr, int K, SumSqSmem &sm)
{
    const int nq = K >> 2;
    uint32_t mbits = 0u;
    for (int i = threadIdx.x; i < nq; i += kThreads) max_chunk_bits(__ldg(xr + i), mbits);
    const uint32_t E = block_emax(mbits, sm);
    FixedAcc acc;
    if (E < 255u)  // else the row holds an infinity or a NaN: the sum is decided by sm.nonfinite
        for (int i = threadIdx.x; i < nq; i += kThreads) add_chunk_fixed(__ldg(xr + i), E, acc);
    unsigned long long lo, hi;
    fixed_total(acc, lo, hi);
    return block_sum_squares(lo, hi, acc.sticky, E, xr, K, sm);
}

// The same from the row's chunks already in registers (v[j] = chunk
// threadIdx.x + j kThreads, valid below nq).
__device__ double row_sum_squares_regs(const float4 (&v)[kRegChunks], const float4 *__restrict__ xr, int K,
                                       SumSqSmem &sm)
{
    const int nq = K >> 2;
    uint32_t mbits = 0u;
#pragma unroll
    for (int j = 0; j < kRegChunks; ++j)
        if (static_cast<int>(threadIdx.x) + j * kThreads < nq) max_chunk_bits(v[j], mbits);
    const uint32_t E = block_emax(mbits, sm);
    FixedAcc acc;
    if (E < 255u) {  // else the row holds an infinity or a NaN: the sum is decided by sm.nonfinite
#pragma unroll
        for (int j = 0; j < kRegChunks; ++j)
            if (static_cast<int>(threadIdx.x) + j * kThreads < nq) add_chunk_fixed(v[j], E, acc);
    }
    unsigned long long lo, hi;
    fixed_total(acc, lo, hi);
    return block_sum_squares(lo, hi, acc.sticky, E, xr, K, sm);
}

// Q8_0 of the normalized chunk x4 (one of the eight chunks of its 32-block,
// the eight lanes of a block being adjacent): the packed codes and, from
// every lane, the block's d.  All lanes of the warp take part (shuffles).
__device__ __forceinline__ uint32_t quant_chunk(float4 x4, float4 w4, float inv, float offset, bool active,
                                                float &d)
{
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    if (active) {
        e[0] = __fmul_rn(__fmul_rn(x4.x, inv), __fadd_rn(w4.x, offset));
        e[1] = __fmul_rn(__fmul_rn(x4.y, inv), __fadd_rn(w4.y, offset));
        e[2] = __fmul_rn(__fmul_rn(x4.z, inv), __fadd_rn(w4.z, offset));
        e[3] = __fmul_rn(__fmul_rn(x4.w, inv), __fadd_rn(w4.w, offset));
    }
    float amax = fmaxf(fmaxf(fabsf(e[0]), fabsf(e[1])), fmaxf(fabsf(e[2]), fabsf(e[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    d = __fdiv_rn(amax, 127.0f);
    return q8_pack4(e, d);
}

// inv = f32(1 / sqrt(ss / K + eps)) in double, each operation rounded to
// nearest, computed by one thread (the double pipe is a small fraction of the
// f32 one on this part) and returned to every thread.
__device__ __forceinline__ float block_inv_rms(double ss, int K, float eps, SumSqSmem &sm)
{
    if (threadIdx.x == 0) {
        const double r = __dsqrt_rn(__dadd_rn(__ddiv_rn(ss, static_cast<double>(K)), static_cast<double>(eps)));
        sm.inv = __double2float_rn(__ddiv_rn(1.0, r));
    }
    __syncthreads();
    return sm.inv;
}

__global__ void __launch_bounds__(kThreads)
    k_rmsnorm_q8_0(const float4 *__restrict__ X, const float4 *__restrict__ w, float offset, float eps,
                   uint32_t *__restrict__ Xq, float *__restrict__ dx, int K)
{
    __shared__ SumSqSmem sm;
    const int t = blockIdx.x;
    const int nblk = K >> 5;
    const float4 *xr = X + static_cast<size_t>(t) * (K >> 2);
    const int nq = K >> 2;
    uint32_t *qr = Xq + static_cast<size_t>(t) * (nblk * 8);
    float *dr = dx + static_cast<size_t>(t) * nblk;
    if (nq <= kRegChunks * kThreads) {
        // the norm weights never depend on the previous kernel: ask L2 for
        // them before waiting (K * 4 bytes, a multiple of 128)
        if (threadIdx.x == 0) prefetch_l2_bulk(w, static_cast<uint32_t>(K) * 4u);
        // dependents launch once every CTA has started; they still wait for
        // this grid's completion before reading Xq and dx
        pdl_launch_dependents();
        pdl_wait();
        // the row is read once: chunk i = threadIdx.x + j kThreads is v[j];
        // the eight chunks of a 32-block sit in eight adjacent lanes
        float4 v[kRegChunks];
#pragma unroll
        for (int j = 0; j < kRegChunks; ++j) {
            const int i = static_cast<int>(threadIdx.x) + j * kThreads;
            v[j] = i < nq ? __ldg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const double ss = row_sum_squares_regs(v, xr, K, sm);
        const float inv = block_inv_rms(ss, K, eps, sm);
#pragma unroll
        for (int j = 0; j < kRegChunks; ++j) {
            const int i = static_cast<int>(threadIdx.x) + j * kThreads;
            if (j * kThreads >= nq) break;  // warp-uniform (kThreads is a multiple of 32)
            const bool active = i < nq;
            const float4 w4 = active ? __ldg(w + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            float d;
            const uint32_t packed = quant_chunk(v[j], w4, inv, offset, active, d);
            if (active) {
                qr[i] = packed;
                if ((i & 7) == 0) dr[i >> 3] = d;
            }
        }
        return;
    }
    pdl_launch_dependents();
    pdl_wait();
    const double ss = row_sum_squares(xr, K, sm);
    const float inv = block_inv_rms(ss, K, eps, sm);

    // Q8_0 of y: eight lanes per 32-block (four elements each), four blocks
    // per warp in a warp-uniform loop so the full-mask shuffles never diverge
    const int sub = threadIdx.x & 7;
    for (int wb = (threadIdx.x >> 5) * 4; wb < nblk; wb += (kThreads >> 5) * 4) {
        const int blk = wb + ((threadIdx.x & 31) >> 3);
        const bool active = blk < nblk;
        const float4 x4 = active ? xr[blk * 8 + sub] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 w4 = active ? __ldg(w + blk * 8 + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
        float d;
        const uint32_t packed = quant_chunk(x4, w4, inv, offset, active, d);
        if (active) {
            qr[blk * 8 + sub] = packed;
            if (sub == 0) dr[blk] = d;
        }
    }
}

// The statistic alone: ss[t] for every row (for tests of the exact sum).
__global__ void __launch_bounds__(kThreads) k_row_sum_squares(const float4 *__restrict__ X, double *__restrict__ ss, int K)
{
    __shared__ SumSqSmem sm;
    pdl_launch_dependents();
    pdl_wait();
    const double v = row_sum_squares(X + static_cast<size_t>(blockIdx.x) * (K >> 2), K, sm);
    if (threadIdx.x == 0) ss[blockIdx.x] = v;
}

}  // namespace norm

int launch_row_sum_squares(const float *X, double *ss, int K, int M, cudaStream_t s)
{
    return status_from(launch_pdl(norm::k_row_sum_squares, dim3(static_cast<unsigned>(M)), dim3(norm::kThreads), 0, s,
                                  reinterpret_cast<const float4 *>(X), ss, K));
}

int launch_rmsnorm_q8_0(const float *X, const float *w, float offset, float eps, int8_t *Xq, float *dx, int K,
                        int M, cudaStream_t s)
{
    return status_from(launch_pdl(norm::k_rmsnorm_q8_0, dim3(static_cast<unsigned>(M)), dim3(norm::kThreads), 0, s,
                                  reinterpret_cast<const float4 *>(X), reinterpret_cast<const float4 *>(w), offset,
                                  eps, reinterpret_cast<uint32_t *>(Xq), dx, K));
}

}  // namespace gq
