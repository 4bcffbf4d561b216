// gq_logits.cu -- Q8_0 tied-embedding logits with soft-cap and on-GPU top-k.
//
// "Gemma 4 M4 Max kernel roadmap": K1 (logit soft-capping), K2 step 6 (final
// Q8_0 embedding/output projection and on-GPU top-k reduction), K5 (a
// pair-valued (value, token) frontier instead of gathering full logits;
// exact truncation of every merge to k pairs).
//
// One kernel (k_q8_0_logits_topk): the Q8_0 matvec core; each warp soft-caps
// its rows' logits, optionally stores them, and keeps the k best (value, row)
// keys it has seen in a warp-resident sorted list; each CTA then merges its
// warps' lists and writes k keys to the workspace.  The last CTA to finish
// (a counter at the start of the workspace, incremented with wrap-around so
// it is back at zero after every call) merges all CTA lists: every key that
// can still be in the final top k is at least the largest k-th key of any
// CTA list (that list alone holds k keys above it) and at least the k-th
// largest list head (the k best heads are k keys above it), so only the
// lists whose head reaches the larger of the two bounds are read, and only
// their keys above it are merged.  (A separate one-CTA merge kernel cost
// 14.7 us per call at 262144 x 5376, against 234 us for the whole stream.)
#include "gq_host.h"
#include "gq_matvec.cuh"

namespace gq {

// The workspace starts with a 16-byte header (the finished-CTA counter),
// then one list of k keys per CTA.
constexpr size_t kLogitsWsHeaderWords = 2;

// Insert every key of `key` (one per lane; 0 = none) that beats the list's
// admission threshold; thr never drops below floor_thr.
__device__ __forceinline__ void offer(WarpTopK &top, unsigned long long &thr, unsigned long long floor_thr,
                                      unsigned long long key, int k)
{
    unsigned int want = __ballot_sync(0xffffffffu, key > thr);
    while (want) {
        const int src = __ffs(want) - 1;
        want &= want - 1;
        const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
        if (kk > thr) {
            top.insert(kk, k);
            const unsigned long long t = top.kth(k);
            thr = t > floor_thr ? t : floor_thr;
        }
    }
}

template <int LG, int R, int U>
__global__ void __launch_bounds__(kThreadsPerCta, 2)
    k_q8_0_logits_topk(const uint4 *__restrict__ qb, const uint16_t *__restrict__ dsc,
                       const float *__restrict__ x, float softcap, int k,
                       float *__restrict__ logits, unsigned long long *__restrict__ ws, int *__restrict__ idx,
                       float *__restrict__ val, int rows, int nb)
{
    extern __shared__ __align__(16) float xs[];
    __shared__ __align__(16) unsigned long long cta_keys[kWarpsPerCta * GQ_MAX_TOPK];
    __shared__ unsigned long long wmax[kWarpsPerCta];
    __shared__ int s_last;
    __shared__ unsigned long long s_t2;
    // Candidates for a merge: every key >= the merge's threshold, gathered in
    // shared memory and sorted by one warp (the usual case: at most k keys
    // per list can reach the threshold, and only a few lists do).
    constexpr int kMaxCand = 128;
    __shared__ unsigned long long cand[kMaxCand];
    __shared__ int s_cnt;
    unsigned int *counter = reinterpret_cast<unsigned int *>(ws);
    unsigned long long *keys = ws + kLogitsWsHeaderWords;
    constexpr int G = 32 / LG, TR = G * R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    auto gather_candidate = [&](unsigned long long key, unsigned long long T) {
        if (key != 0ull && key >= T) {
            const int pos = atomicAdd(&s_cnt, 1);
            if (pos < kMaxCand) cand[pos] = key;
        }
    };
    // warp-wide: the s_cnt candidates sorted descending, entry i in
    // e[i / 32] of lane i % 32 (entries past s_cnt are 0)
    auto sort_candidates = [&](unsigned long long (&e)[4]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = lane + 32 * j;
            e[j] = i < s_cnt ? cand[i] : 0ull;
        }
        warp_sort128_desc(e);
    };
    const int g = lane / LG, lp = lane % LG;
    const int ntasks = (rows + TR - 1) / TR;
    const bool cap = softcap > 0.f;
    const int first = blockIdx.x * kWarpsPerCta + warp;

    if (first < ntasks) {
        const void *rp[TR];
#pragma unroll
        for (int i = 0; i < TR; ++i) rp[i] = qb + static_cast<size_t>(min(first * TR + i, rows - 1)) * nb * 2;
        prefetch_rows_l2<TR>(rp, static_cast<uint32_t>(nb) * 32u, lane);
    }
    pdl_wait();
    stage_x(xs, x, nb * 32);
    pdl_launch_dependents();

    WarpTopK top;
    top.init();
    unsigned long long thr = 0ull;

    for (int task = first; task < ntasks; task += gridDim.x * kWarpsPerCta) {
        const int r0 = task * TR + g * R;
        const uint4 *wp[R];
        const uint16_t *sp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = min(r0 + i, rows - 1);
            wp[i] = qb + static_cast<size_t>(r) * nb * 2;
            sp[i] = dsc + static_cast<size_t>(r) * nb;
        }
        float out[R];
        q8_0_stream<LG, R, U>(wp, sp, xs, nb, lp, out);
        // lane lp < R of a group keeps row r0 + lp: one soft-cap per lane and
        // one offer per task cover all of the task's rows
        static_assert(R <= LG, "a group needs a lane per row");
        float l = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float v = group_sum<LG>(out[i]);
            if (lp == i) l = v;
        }
        const int r = r0 + lp;
        const bool mine = lp < R && r < rows;
        if (cap) l = softcap * tanhf(__fdiv_rn(l, softcap));
        if (mine && logits != nullptr) logits[r] = l;
        offer(top, thr, 0ull, mine ? topk_key(l, static_cast<uint32_t>(r)) : 0ull, k);
    }

    // merge the warps' lists (lane j holds entry j in e0 and entry j+32 in e1)
    for (int j = lane; j < k; j += 32) cta_keys[warp * k + j] = (j < 32) ? top.e0 : top.e1;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    {
        // every key of this CTA's top k is >= the largest k-th key of a warp list
        unsigned long long T = 0ull;
#pragma unroll
        for (int w = 0; w < kWarpsPerCta; ++w) {
            const unsigned long long v = cta_keys[w * k + k - 1];
            T = v > T ? v : T;
        }
        for (int j = threadIdx.x; j < kWarpsPerCta * k; j += kThreadsPerCta) gather_candidate(cta_keys[j], T);
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long e[4];
        if (s_cnt <= kMaxCand) {
            sort_candidates(e);
        } else {  // more than kMaxCand keys at or above the threshold (ties): insert one by one
            top.init();
            thr = 0ull;
            for (int base = 0; base < kWarpsPerCta * k; base += 32) {
                const int j = base + lane;
                offer(top, thr, 0ull, (j < kWarpsPerCta * k) ? cta_keys[j] : 0ull, k);
            }
            e[0] = top.e0;
            e[1] = top.e1;
        }
        if (lane < k) keys[static_cast<size_t>(blockIdx.x) * k + lane] = e[0];
        if (lane + 32 < k) keys[static_cast<size_t>(blockIdx.x) * k + lane + 32] = e[1];
        // this CTA's keys are visible device-wide before it counts itself
        __threadfence();
        __syncwarp();
        if (lane == 0) s_last = atomicInc(counter, gridDim.x - 1) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // and the other CTAs' keys are visible here

    // ---- the last CTA: merge all CTA lists (keys read through L2; every list
    // is sorted, largest first).  Two lower bounds on the final k-th key:
    //   T1, the largest k-th key of any list (that list alone holds k keys
    //       at or above it);
    //   T2, the k-th largest list head (those k heads are k distinct keys at
    //       or above it), usually far higher: with hundreds of similar lists
    //       T1 lets a large fraction of all keys through.
    // Only lists whose head reaches T = max(T1, T2) are read further.
    const int nlists = gridDim.x;
    unsigned long long t = 0ull;
    for (int c = threadIdx.x; c < nlists; c += kThreadsPerCta) {
        const unsigned long long v = __ldcg(keys + static_cast<size_t>(c) * k + (k - 1));
        t = v > t ? v : t;
        if (nlists <= kWarpsPerCta * GQ_MAX_TOPK) cta_keys[c] = __ldcg(keys + static_cast<size_t>(c) * k);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long v = __shfl_xor_sync(0xffffffffu, t, o);
        t = v > t ? v : t;
    }
    if (lane == 0) wmax[warp] = t;
    if (threadIdx.x == 0) {
        s_cnt = 0;
        s_t2 = 0ull;
    }
    __syncthreads();
    if (nlists <= kWarpsPerCta * GQ_MAX_TOPK && nlists >= k) {
        // rank of each head among all heads, from pairs of heads in four
        // independent counts (a zero pads an odd count: it is above no key);
        // keys are unique apart from 0 (an empty entry), whose rank-(k-1)
        // writers all write 0
        if (threadIdx.x == 0 && (nlists & 1)) cta_keys[nlists] = 0ull;
        __syncthreads();
        const ulonglong2 *hp = reinterpret_cast<const ulonglong2 *>(cta_keys);
        const int npairs = (nlists + 1) >> 1;
        for (int c = threadIdx.x; c < nlists; c += kThreadsPerCta) {
            const unsigned long long h = cta_keys[c];
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
            int j = 0;
            for (; j + 1 < npairs; j += 2) {
                const ulonglong2 a = hp[j], b = hp[j + 1];
                r0 += a.x > h ? 1 : 0;
                r1 += a.y > h ? 1 : 0;
                r2 += b.x > h ? 1 : 0;
                r3 += b.y > h ? 1 : 0;
            }
            if (j < npairs) {
                const ulonglong2 a = hp[j];
                r0 += a.x > h ? 1 : 0;
                r1 += a.y > h ? 1 : 0;
            }
            if (r0 + r1 + r2 + r3 == k - 1) s_t2 = h;
        }
        __syncthreads();
    }
    unsigned long long T = s_t2;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) T = wmax[w] > T ? wmax[w] : T;
    const unsigned long long floor_thr = T > 0ull ? T - 1ull : 0ull;  // admit keys >= T
    const int nkeys = nlists * k;
    // gather the candidates (keys >= T) from the lists whose head reaches T,
    // eight keys of a list per batch of loads
    constexpr int kBatch = 4;
    for (int c = threadIdx.x; c < nlists; c += kThreadsPerCta) {
        const unsigned long long *lst = keys + static_cast<size_t>(c) * k;
        if (__ldcg(lst) < T) continue;
        for (int j0 = 0; j0 < k; j0 += 8) {
            unsigned long long kk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) kk[u] = (j0 + u < k) ? __ldcg(lst + j0 + u) : 0ull;
            bool more = true;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                gather_candidate(kk[u], T);
                more = more && kk[u] >= T;
            }
            if (!more) break;
        }
    }
    __syncthreads();
    unsigned long long e[4];
    if (s_cnt <= kMaxCand) {
        if (warp != 0) return;
        sort_candidates(e);
    } else {
        // more than kMaxCand keys at or above the threshold (ties): per-warp
        // insertion, then warp 0 merges the warp lists
        top.init();
        thr = floor_thr;
        for (int base = warp * 32; base < nkeys; base += kBatch * kThreadsPerCta) {
            unsigned long long kk[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = base + u * kThreadsPerCta + lane;
                kk[u] = (j < nkeys) ? __ldcg(keys + j) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) offer(top, thr, floor_thr, kk[u], k);
        }
        for (int j = lane; j < k; j += 32) cta_keys[warp * k + j] = (j < 32) ? top.e0 : top.e1;
        __syncthreads();
        if (warp != 0) return;
        top.init();
        thr = floor_thr;
        for (int base = 0; base < kWarpsPerCta * k; base += 32) {
            const int j = base + lane;
            offer(top, thr, floor_thr, (j < kWarpsPerCta * k) ? cta_keys[j] : 0ull, k);
        }
        e[0] = top.e0;
        e[1] = top.e1;
    }
    if (lane < k) {
        idx[lane] = static_cast<int>(key_row(e[0]));
        val[lane] = key_value(e[0]);
    }
    if (lane + 32 < k) {
        idx[lane + 32] = static_cast<int>(key_row(e[1]));
        val[lane + 32] = key_value(e[1]);
    }
}

// Upper bound on the CTAs of the logits kernels, fixed so the workspace size
// depends only on the arguments, not on the GPU.
constexpr int kLogitsMaxCtas = 2048;
int logits_max_ctas() { return kLogitsMaxCtas; }

size_t logits_topk_ws_bytes(int rows, int K, int k)
{
    (void)K;
    const long long tasks_ctas = (static_cast<long long>(rows) + 7) / 8;
    const long long ctas = tasks_ctas < kLogitsMaxCtas ? tasks_ctas : kLogitsMaxCtas;
    return (kLogitsWsHeaderWords + static_cast<size_t>(ctas) * static_cast<size_t>(k)) * sizeof(unsigned long long);
}

int launch_logits_topk(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                       float *logits, void *ws, size_t ws_bytes, int rows, int K, MatvecGeo geo,
                       cudaStream_t s)
{
    const int nb = K / 32;
    const uint4 *qb = static_cast<const uint4 *>(W);
    const uint16_t *dsc = reinterpret_cast<const uint16_t *>(qb + static_cast<size_t>(rows) * nb * 2);
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    const long long ntasks = (rows + (32 / geo.lg) * geo.r - 1) / ((32 / geo.lg) * geo.r);
    unsigned long long *wsw = static_cast<unsigned long long *>(ws);
#define CASE(LG, R, U)                                                                                 \
    {                                                                                                  \
        auto kern = k_q8_0_logits_topk<LG, R, U>;                                                      \
        int grid = persistent_grid(reinterpret_cast<const void *>(kern), kThreadsPerCta, smem, ntasks); \
        if (grid <= 0) return GQ_ERR_SHAPE;                                                            \
        if (grid > kLogitsMaxCtas) grid = kLogitsMaxCtas;                                              \
        if ((kLogitsWsHeaderWords + static_cast<size_t>(grid) * k) * sizeof(unsigned long long) > ws_bytes) \
            return GQ_ERR_WORKSPACE;                                                                   \
        return status_from(launch_pdl(kern, dim3(grid), dim3(kThreadsPerCta), smem, s, qb, dsc, x, softcap, k, \
                                      logits, wsw, idx, val, rows, nb));                               \
    }
    GQ_GEO_SWITCH(geo, CASE);
#undef CASE
}

}  // namespace gq
