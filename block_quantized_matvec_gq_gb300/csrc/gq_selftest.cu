// gq_selftest.cu -- a check of the bounded-wait path every tensor-core
// kernel relies on: one thread waits on an mbarrier whose phase nothing
// completes, through the same wait helper and time limit as the kernels;
// the wait gives up, records GQ_ERR_TIMEOUT in the device status word and
// the kernel returns normally (no fault; the context stays usable).
#include "gq_tc.cuh"

namespace gq {

__global__ void k_selftest_bounded_wait(int *__restrict__ status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tcu::mbar_init(tcu::smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int *ab = &abort_flag;
        tcu::wait_bounded(tcu::smem_u32(&bar), 0u, ab, status);  // phase 0 never completes
    }
}

int launch_selftest_bounded_wait(cudaStream_t s)
{
    int *st = status_word();
    if (st == nullptr) return GQ_ERR_CUDA;
    k_selftest_bounded_wait<<<1, 32, 0, s>>>(st);
    return status_from(cudaGetLastError());
}

}  // namespace gq
