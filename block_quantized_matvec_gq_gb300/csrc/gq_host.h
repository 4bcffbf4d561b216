// gq_host.h -- host-side helpers shared by the libgq launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gq.h"

namespace gq {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

inline int status_from(cudaError_t e) { return e == cudaSuccess ? GQ_OK : GQ_ERR_CUDA; }

// Streaming multiprocessor count of the current device (cached per device).
inline int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

// Resident CTAs per SM for (kernel, threads, dynamic smem), cached.  The
// first time a kernel is seen on a device its dynamic shared-memory limit is
// raised to the device's opt-in maximum (once: lowering it again for a
// smaller launch would break a later larger one).
inline int ctas_per_sm(const void *kern, int threads, size_t smem)
{
    struct Entry {
        const void *k;
        int dev, threads;
        size_t smem;
        int occ;
    };
    struct Raised {
        const void *k;
        int dev;
    };
    static Entry tab[512];
    static Raised raised[256];
    static int used = 0, nraised = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (tab[i].k == kern && tab[i].dev == dev && tab[i].threads == threads && tab[i].smem == smem)
            return tab[i].occ;
    bool done = false;
    for (int i = 0; i < nraised; ++i)
        if (raised[i].k == kern && raised[i].dev == dev) done = true;
    if (!done) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa;
        const size_t static_smem = (cudaFuncGetAttributes(&fa, kern) == cudaSuccess) ? fa.sharedSizeBytes : 0;
        const int maxdyn = optin - static_cast<int>(static_smem);
        if (maxdyn > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, maxdyn);
        cudaGetLastError();  // never leave an error behind for a later launch check
        if (nraised < 256) raised[nraised++] = Raised{kern, dev};
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem) != cudaSuccess) {
        cudaGetLastError();  // clear: an unfit configuration is reported as occ = 0
        occ = 0;
    }
    if (used < 512) tab[used++] = Entry{kern, dev, threads, smem, occ};
    return occ;
}

// Persistent grid: enough CTAs for ntasks warp tasks, at most SMs x resident CTAs.
inline int persistent_grid(const void *kern, int threads, size_t smem, long long ntasks)
{
    const int occ = ctas_per_sm(kern, threads, smem);
    if (occ <= 0) return -1;
    const int warps = threads / 32;
    const long long want = (ntasks + warps - 1) / warps;
    const long long cap = static_cast<long long>(sm_count()) * occ;
    return static_cast<int>(want < cap ? want : cap);
}

// Launch with programmatic stream serialization allowed (the kernel itself
// calls griddepcontrol.wait before it reads anything a previous kernel wrote).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- internal launchers
// Matvec geometry: LG lanes per row group, R rows per group, U blocks in flight.
struct MatvecGeo {
    int lg, r, u, warps;
};

MatvecGeo choose_matvec_geo(int format, int rows, int nb, bool pair_ok);
MatvecGeo choose_logits_geo(int rows, int nb);
MatvecGeo choose_ffn_geo(int rows, int nb, bool pair_ok);
MatvecGeo choose_q6k_geo();

int launch_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo g,
                       cudaStream_t s);
int launch_q8_0_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo g,
                       cudaStream_t s);
int launch_q6k_matvec(const void *W, const float *x, float *y, int rows, int K, cudaStream_t s);
int launch_selftest_bounded_wait(cudaStream_t s);
int launch_q4k_matvec(const void *W, const float *x, float *y, int rows, int K, MatvecGeo g,
                      cudaStream_t s);
int launch_ffn_gate_up(const void *Wg, const void *Wu, const float *x, float *h, int rows, int K,
                       MatvecGeo g, cudaStream_t s);
size_t logits_topk_ws_bytes(int rows, int K, int k);
int launch_logits_topk(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                       float *logits, void *ws, size_t ws_bytes, int rows, int K, MatvecGeo g,
                       cudaStream_t s);

int launch_pack(int format, const void *src, void *dst, int rows, int K, bool unpack,
                cudaStream_t s);
int launch_quantize_q8_0(const float *X, int8_t *Xq, float *dx, int K, int M, cudaStream_t s);
size_t gemm_workspace_bytes(int K, int M);
// scale-folded bf16 tensor-core path (gq_gemm_split.cu): K % 256 == 0
size_t gemm_split_workspace_bytes(int K, int M);
bool gemm_split_supported(int K);
bool gemm_small_supported(int K, int M);
// register-operand tensor-core path with exact block dots (gq_gemm_mma.cu): K % 256 == 0
bool gemm_mma_supported(int K, int M);
size_t gemm_mma_workspace_bytes(int K, int M);
int gemm_mma_max_tokens();
int launch_gemm_mma(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes, int rows,
                    int K, int M, cudaStream_t s);
int launch_gemm_small(const void *W, const int8_t *Xq, const float *dx, float *Y, int rows, int K, int M,
                      cudaStream_t s);
int launch_gemm_split(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes,
                      int rows, int K, int M, cudaStream_t s);
int launch_gemm_q8act_tc(const void *W, const int8_t *Xq, const float *dx, float *Y, void *ws, size_t ws_bytes,
                         int rows, int K, int M, cudaStream_t s);
int launch_block_dots_tc(const void *W, const int8_t *Xq, int32_t *D, void *ws, size_t ws_bytes, int rows, int K,
                         int M, cudaStream_t s);
// ring-streamed 4-bit matvecs (gq_stream.cu)
bool ring_preferred(int rows, int nb);
int schedule_mode(long long ntasks, long long warps, int nb);
bool gemm_force_block_path();
bool ring_q4_0_supported(int nb);
int launch_ring_q4_0(const void *W, const float *x, const float *g_or_null, const float *u, float *y, int rows,
                     int K, cudaStream_t s);
int launch_ring_ffn(const void *Wg, const void *Wu, const float *x, float *h, int rows, int K, cudaStream_t s);
int launch_ring_q4k(const void *W, const float *x, float *y, int rows, int K, cudaStream_t s);
int read_device_status(bool reset);
int *status_word();  // device address of the status word (current device)

}  // namespace gq
