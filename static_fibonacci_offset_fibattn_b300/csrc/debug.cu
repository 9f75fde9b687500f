// debug.cu -- a check of the failure path: one wait that runs out.
//
// Every wait of the attention kernels is bounded (tc::mbar_wait): on expiry it latches the
// device error word, the kernel tears down (its TMEM released) and returns, and the host
// reads the status with fibattn_poll_device_error. This kernel waits, with the same bounded
// wait, on an mbarrier that nothing arrives on, so a test can see that path end in a TIMEOUT
// status with the context still usable -- without a fault, a trap or a hang.
#include <stdint.h>

#include "internal.h"
#include "tc_prims.cuh"

namespace fibattn {
namespace {

__global__ void wait_timeout_kernel(int32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);  // one arrival expected, none will come
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        bool aborted = false;
        tc::mbar_wait(b, 0, aborted, err, limit_ns);
    }
}

}  // namespace
}  // namespace fibattn

using namespace fibattn;

extern "C" fibattn_status fibattn_debug_wait_timeout(int32_t limit_ms, void* cuda_stream) {
    if (limit_ms < 1 || limit_ms > 10000) return FIBATTN_ERR_INVALID_ARG;
    int32_t* err = device_error_word();
    if (!err) return cuda_fail(-1, "cudaGetSymbolAddress (error word)");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    {
        KernelScope ks("debug_wait_timeout", st);
        wait_timeout_kernel<<<1, 32, 0, st>>>(err, (uint64_t)limit_ms * 1000000ull);
    }
    return launch_status("launch debug_wait_timeout");
}
