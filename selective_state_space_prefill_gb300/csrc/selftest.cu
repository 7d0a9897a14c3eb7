// selftest.cu -- a diagnostic kernel that lets a caller watch the library's bounded-wait
// machinery fail safely: it waits on an mbarrier phase that nothing completes, through the
// same bounded wait the TMA pipelines use, and reports the expiry in the device status word
// (SSM_DEV_WAIT_TIMEOUT) before returning normally.  No trap, no fault, no unbounded spin.
#include "common.cuh"
#include "kernels.h"

namespace ssm {
namespace {

__global__ void k_expire_wait(unsigned int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);                 // one arrival expected; none ever comes
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, limit_ns)) atomicOr(status, 1u);
}

}  // namespace

int launch_expire_wait(unsigned int* status, uint64_t limit_ns, cudaStream_t stream, const char** why) {
    k_expire_wait<<<1, 32, 0, stream>>>(status, limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return -1;
    }
    return 0;
}

}  // namespace ssm
