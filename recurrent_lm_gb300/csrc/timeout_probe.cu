// la_debug_timeout_probe: exercises the bounded-wait failure path on the GPU
// without a fault.  One thread waits, through the same bounded mbarrier wait
// that every kernel of the library uses, on a barrier phase that nothing
// completes.  After the wait's limit (about one second) it records a timeout
// in the device status word and the kernel returns, leaving the context
// usable; la_check_device_status then reports LA_ERR_TIMEOUT.
#include "la_internal.h"
#include "tc_common.cuh"

namespace la {
namespace {

__global__ void timeout_probe_kernel(unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(tc::smem_u32(&bar), 1);
        abort_flag = 0;
        tc::mbar_init_fence();
    }
    __syncthreads();
    // phase 0 never completes: no thread arrives on the barrier
    if (threadIdx.x == 0) (void)tc::mbar_wait(tc::smem_u32(&bar), 0u, &abort_flag, status);
}

}  // namespace

cudaError_t launch_timeout_probe(unsigned *status, cudaStream_t st) {
    timeout_probe_kernel<<<1, 32, 0, st>>>(status);
    return cudaGetLastError();
}

}  // namespace la
