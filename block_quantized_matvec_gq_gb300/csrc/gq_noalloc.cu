// gq_noalloc.cu -- the tied-logit top-k for callers that cannot allocate.
//
// gq_logits_topk needs a device workspace for its per-CTA key lists.  Some
// callers cannot provide one: a serving loop that must never call
// cudaMalloc once it runs (the call can synchronize the device), or a host
// runtime that only passes the library its input and output buffers.  This
// entry point keeps the key lists in a fixed array of the library's own
// device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU on which the
// library is loaded holds it (1 MiB) until the process exits.  In host code
// its name is only a host-side stand-in, never a device address: the device
// address is looked up once per device with cudaGetSymbolAddress (on the
// first call made with that device current) and passed to the kernels.
// All calls share the array: two calls whose kernels may overlap on the GPU
// (different streams without ordering) race on it.  Its counter starts at
// zero (static device memory is zero-initialised) and every completed call
// leaves it at zero; every key a call reads was written earlier in that call.
#include "gq_host.h"

namespace gq {

// A 16-byte header (the finished-CTA counter, zero at load and back at zero
// after every call) and one list of up to GQ_MAX_TOPK keys for each of up
// to 2048 CTAs: every call that gq_logits_topk accepts fits.
constexpr size_t kNoallocScratchWords = 2 + 2048ull * GQ_MAX_TOPK;
constexpr size_t kNoallocScratchBytes = kNoallocScratchWords * sizeof(unsigned long long);

static __device__ __align__(256) unsigned long long g_topk_scratch[kNoallocScratchWords];

// Device address of the scratch array on the current device (looked up once
// per device); nullptr if the lookup fails.
static void *topk_scratch_address()
{
    static void *cache[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = p;
    }
    return cache[dev];
}

}  // namespace gq

extern "C" int gq_logits_topk_noalloc(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                                      float *logits_or_null, int rows, int K, int M, gq_stream_t stream)
{
    const size_t need = gq_logits_topk_workspace_bytes(rows, K, k);
    if (need == 0) return GQ_ERR_SHAPE;                          // k or rows out of range
    if (need > gq::kNoallocScratchBytes) return GQ_ERR_SHAPE;    // beyond the fixed array
    void *ws = gq::topk_scratch_address();
    if (ws == nullptr) return GQ_ERR_CUDA;
    return gq_logits_topk(W, x, softcap, k, idx, val, logits_or_null, ws, gq::kNoallocScratchBytes, rows, K, M,
                          stream);
}
