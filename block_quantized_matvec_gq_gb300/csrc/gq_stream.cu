// gq_stream.cu -- host side of the ring-streamed 4-bit decode matvecs
// (gq_ring.cuh): the Q4_0 matvec, the Q4_0 down projection with the GELU
// gate formed while staging, the fused Q4_0 gate/up pair, and the Q4_K
// matvec.
//
// "Gemma 4 M4 Max kernel roadmap", K2 "Metal decode path" (direct Q4_0
// matrix-vector product with fused dequantization and F32 accumulation;
// the gated GELU projection pair) and K5 (exact gate/up launch fusion);
// "Metal kernel capability table (Phase B ground truth)", section 1
// (q4_f32_matvec, q4k_matvec: rows masked, K checked at dispatch), section 4
// (the clamped GELU-tanh of the gated FFN and of the fused down kernels) and
// section 8 (K-alignment and tail hazards: K is never truncated; a short,
// wide matrix is split along K and its partial sums added in a fixed order).
#include <stdlib.h>

#include "gq_host.h"
#include "gq_ring.cuh"

namespace gq {

namespace {

using ring::Plan;

constexpr int kSmemLimit = 227 * 1024;

// Geometry of one launch (the compile-time part selects the instantiation).
struct RingGeo {
    int r = 2;      // rows per lane group (rows per stage = 4 r)
    int w = 16;     // warps per CTA
    int s = 2;      // stages per warp
    int kc = 32;    // K units per stage chunk
    int cs = 0;     // CTAs per cluster (0: chosen by shape)
};

#ifdef GQ_TUNING
// Geometry sweeps: a tuning build reads overrides from the environment.
void tuning_override(RingGeo &g)
{
    if (const char *v = getenv("GQ_RING_R")) g.r = atoi(v);
    if (const char *v = getenv("GQ_RING_W")) g.w = atoi(v);
    if (const char *v = getenv("GQ_RING_S")) g.s = atoi(v);
    if (const char *v = getenv("GQ_RING_KC")) g.kc = atoi(v);
    if (const char *v = getenv("GQ_RING_CS")) g.cs = atoi(v);
}
#else
void tuning_override(RingGeo &) {}
#endif

int max_active_clusters(const void *kern, int threads, int cs, size_t smem)
{
    struct Entry {
        const void *k;
        int dev, cs;
        size_t smem;
        int n;
    };
    static Entry tab[256];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (tab[i].k == kern && tab[i].dev == dev && tab[i].cs == cs && tab[i].smem == smem) return tab[i].n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs * 64);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (used < 256) tab[used++] = Entry{kern, dev, cs, smem, n};
    return n;
}

// Shared memory of one CTA: the staged x slice, the ring, the cluster sums.
struct Layout {
    int cs, ncl;
    Plan p;
    size_t smem;
};

template <class F>
bool layout(int rows, int nk, int unit, int W, int S, int cs, int ncl, Layout &L)
{
    const int nunits = nk / unit;
    if (cs < 1 || cs > 8 || cs > nunits || ncl < 1) return false;
    const int slice_units = (nunits + cs - 1) / cs;
    const size_t xbytes = static_cast<size_t>(slice_units) * unit * F::kXPerUnit * kXBlk * sizeof(float);
    const size_t ring_off = (xbytes + 127) & ~static_cast<size_t>(127);
    const size_t ring_bytes = static_cast<size_t>(W) * S * F::kStageBytes;
    const size_t red_off = ring_off + ring_bytes;
    const int rows_per_cl = (rows + ncl - 1) / ncl;
    const size_t red_bytes = cs > 1 ? static_cast<size_t>(rows_per_cl) * F::kNM * sizeof(float) : 0;
    const size_t static_bytes = static_cast<size_t>(W) * (S * 8 + W * F::kNR * F::kNM * 4);
    L.smem = red_off + red_bytes;
    if (L.smem + static_bytes > static_cast<size_t>(kSmemLimit)) return false;
    L.cs = cs;
    L.ncl = ncl;
    L.p.unit = unit;
    L.p.cs = cs;
    L.p.ring_off = static_cast<int>(ring_off);
    L.p.red_off = static_cast<int>(red_off);
    return true;
}

template <class F, int R, int W, int S, class In, class Out>
int launch_ring(const typename F::Src &src, In in, Out out, int rows, int nk, int unit, const RingGeo &geo,
                cudaStream_t stream)
{
    auto kern = ring::k_ring_matvec<F, R, W, S, In, Out>;
    constexpr int kThreads = W * 32;
    const void *kp = reinterpret_cast<const void *>(kern);
    int *status = status_word();
    if (status == nullptr) return GQ_ERR_CUDA;
    const int sms = sm_count();
    const int nunits = nk / unit;

    // Every CTA resident at once.  Fewer than four rows per CTA: split K
    // across a cluster so that every CTA keeps at least one row group (four
    // rows) busy.
    Layout L;
    bool ok = false;
    const int want_cl = (rows + 3) / 4;
    int cs = geo.cs;
    if (cs == 0) {
        cs = 1;
        if (want_cl < sms)
            while (cs < 8 && want_cl * cs < sms && cs * 2 <= nunits) cs *= 2;
    }
    for (; cs <= 8 && !ok; cs *= 2) {
        int ncl = cs == 1 ? (want_cl < sms ? want_cl : sms) : 1;
        if (!layout<F>(rows, nk, unit, W, S, cs, ncl, L)) continue;  // the x slice does not fit: split more
        ctas_per_sm(kp, kThreads, L.smem);  // raises the kernel's shared-memory limit once
        if (cs > 1) {
            const int maxcl = max_active_clusters(kp, kThreads, cs, L.smem);
            if (maxcl <= 0) continue;
            ncl = want_cl < maxcl ? want_cl : maxcl;
            if (!layout<F>(rows, nk, unit, W, S, cs, ncl, L)) continue;
        } else {
            // as many CTAs as fit at once (one CTA per SM unless the CTA is small)
            const int occ = ctas_per_sm(kp, kThreads, L.smem);
            if (occ <= 0) continue;
            const int cap = sms * occ;
            L.ncl = want_cl < cap ? want_cl : cap;
        }
        ok = true;
    }
    if (!ok) return GQ_ERR_SHAPE;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.cs * L.ncl);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (L.cs > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = L.cs;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return status_from(cudaLaunchKernelEx(&cfg, kern, src, in, out, rows, nk, L.p, status));
}

// R (rows per lane group), W (warps per CTA), S (stages) and the chunk KC
// are compile-time.
#define GQ_RING_CASE(R_, W_, S_, KC_, ...) \
    if (g.r == R_ && g.w == W_ && g.s == S_ && g.kc == KC_) \
        return launch_ring<__VA_ARGS__, R_, W_, S_, In, Out>(src, in, out, rows, nk, unit, g, s);

template <class In, class Out>
int dispatch_q40x1(const ring::Q40Src<1> &src, In in, Out out, int rows, int nk, int unit, const RingGeo &g,
                   cudaStream_t s)
{
    GQ_RING_CASE(2, 16, 2, 32, ring::Q40<1, 2, 32>)
#ifdef GQ_TUNING
    GQ_RING_CASE(2, 16, 3, 16, ring::Q40<1, 2, 16>)
    GQ_RING_CASE(2, 8, 3, 32, ring::Q40<1, 2, 32>)
    GQ_RING_CASE(2, 8, 2, 64, ring::Q40<1, 2, 64>)
    GQ_RING_CASE(1, 16, 2, 64, ring::Q40<1, 1, 64>)
    GQ_RING_CASE(2, 16, 2, 24, ring::Q40<1, 2, 24>)
#endif
    return GQ_ERR_SHAPE;
}
template <class In, class Out>
int dispatch_q40x2(const ring::Q40Src<2> &src, In in, Out out, int rows, int nk, int unit, const RingGeo &g,
                   cudaStream_t s)
{
    GQ_RING_CASE(1, 16, 2, 32, ring::Q40<2, 1, 32>)
#ifdef GQ_TUNING
    GQ_RING_CASE(2, 16, 2, 16, ring::Q40<2, 2, 16>)
    GQ_RING_CASE(1, 16, 3, 16, ring::Q40<2, 1, 16>)
    GQ_RING_CASE(2, 8, 2, 32, ring::Q40<2, 2, 32>)
    GQ_RING_CASE(1, 16, 2, 24, ring::Q40<2, 1, 24>)
#endif
    return GQ_ERR_SHAPE;
}
template <class In, class Out>
int dispatch_q4k(const ring::Q4KSrc &src, In in, Out out, int rows, int nk, int unit, const RingGeo &g,
                 cudaStream_t s)
{
    GQ_RING_CASE(2, 16, 2, 4, ring::Q4K<2, 4>)
#ifdef GQ_TUNING
    GQ_RING_CASE(2, 16, 3, 2, ring::Q4K<2, 2>)
    GQ_RING_CASE(2, 8, 3, 4, ring::Q4K<2, 4>)
    GQ_RING_CASE(2, 8, 2, 8, ring::Q4K<2, 8>)
    GQ_RING_CASE(1, 16, 2, 8, ring::Q4K<1, 8>)
    GQ_RING_CASE(2, 16, 2, 3, ring::Q4K<2, 3>)
#endif
    return GQ_ERR_SHAPE;
}
#undef GQ_RING_CASE

}  // namespace

// Q4_0 needs whole 8-block groups per row (a row's scales then start on a
// 16-byte boundary, which the bulk copies require).
bool ring_q4_0_supported(int nb) { return nb % 8 == 0; }

int launch_ring_q4_0(const void *W, const float *x, const float *g_or_null, const float *u, float *y, int rows,
                     int K, cudaStream_t s)
{
    const int nb = K / 32;
    ring::Q40Src<1> src;
    src.nib[0] = static_cast<const uint8_t *>(W);
    src.sc[0] = src.nib[0] + static_cast<size_t>(rows) * nb * 16;
    RingGeo geo;
    tuning_override(geo);
    if (g_or_null) return dispatch_q40x1(src, ring::InGeglu{g_or_null, u}, ring::OutY{y}, rows, nb, 8, geo, s);
    return dispatch_q40x1(src, ring::InX{x}, ring::OutY{y}, rows, nb, 8, geo, s);
}

int launch_ring_ffn(const void *Wg, const void *Wu, const float *x, float *h, int rows, int K, cudaStream_t s)
{
    const int nb = K / 32;
    ring::Q40Src<2> src;
    src.nib[0] = static_cast<const uint8_t *>(Wg);
    src.sc[0] = src.nib[0] + static_cast<size_t>(rows) * nb * 16;
    src.nib[1] = static_cast<const uint8_t *>(Wu);
    src.sc[1] = src.nib[1] + static_cast<size_t>(rows) * nb * 16;
    RingGeo geo;
    geo.r = 1;
    tuning_override(geo);
    return dispatch_q40x2(src, ring::InX{x}, ring::OutGeglu{h}, rows, nb, 8, geo, s);
}

int launch_ring_q4k(const void *W, const float *x, float *y, int rows, int K, cudaStream_t s)
{
    const int ns = K / 256;
    ring::Q4KSrc src;
    src.nib = static_cast<const uint8_t *>(W);
    src.rec = src.nib + static_cast<size_t>(rows) * ns * 128;
    RingGeo geo;
    geo.kc = 4;
    tuning_override(geo);
    return dispatch_q4k(src, ring::InXSum{x}, ring::OutY{y}, rows, ns, 1, geo, s);
}

}  // namespace gq
