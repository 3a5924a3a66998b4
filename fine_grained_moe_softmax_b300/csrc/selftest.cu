// selftest.cu -- a probe of the bounded-wait machinery of the pipelined kernels.
//
// One thread waits, with the same wait_phase() the tensor-core GEMM uses, on an mbarrier that
// nothing ever arrives on. The wait gives up after the requested time and records MOE_ERR_TIMEOUT
// in the status word; the kernel then returns normally, so the CUDA context stays usable.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "waits.cuh"

namespace moe {

namespace {

__global__ void bounded_wait_probe_kernel(int* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        wait_phase(ptx::smem_addr(&bar), 0, &abort_flag, status, timeout_ns);
    __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_probe(int* status, uint64_t timeout_ns, cudaStream_t st) {
    bounded_wait_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
