// gq_status.cu -- the device status word that kernels with bounded waits
// report timeouts into (read and cleared by gq_device_status).
#include "gq_host.h"

namespace gq {

static __device__ int g_status_word = 0;

// Device address of the status word on the current device (looked up once
// per device, under a lock: launchers may run on several host threads).
int *status_word()
{
    static int *cache[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

int read_device_status(bool reset)
{
    int *p = status_word();
    if (p == nullptr) return GQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GQ_ERR_CUDA;
    if (reset && v != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return GQ_ERR_CUDA;
    }
    return v;
}

}  // namespace gq
