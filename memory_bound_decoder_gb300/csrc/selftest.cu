// Self-test of the failure path of the bounded waits: a kernel arms an mbarrier for 16 bytes that no peer
// will ever send, so its wait can only end by running out of time. It must give up, set the device error
// bit and return, leaving the context usable.
#include "common.cuh"
#include "launch.h"

namespace mbd {

namespace {

__global__ void bounded_wait_probe(long long limit_cycles) {
    __shared__ Exchange ex;
    if (threadIdx.x == 0) {
        const uint32_t mb = smem_addr(&ex.mbar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 16;" ::"r"(mb) : "memory");
    }
    __syncwarp();
    (void)exchange_wait_warp(ex, limit_cycles);
}

}  // namespace

cudaError_t launch_bounded_wait_probe(long long limit_cycles, cudaStream_t s) {
    bounded_wait_probe<<<1, 32, 0, s>>>(limit_cycles);
    return cudaGetLastError();
}

cudaError_t device_error_flags_selftest(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error_flags, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_flags, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace mbd
