// status.cu -- ABI version and status strings.
#include "pa.h"

extern "C" int pa_abi_version(void) { return 2; }

extern "C" const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

// ---- self-test of the bounded wait ------------------------------------------
#include "pa_device.cuh"

namespace {
// One warp waits on an mbarrier that nothing ever arrives at.  The wait gives
// up after its time limit and reports PA_DERR_TIMEOUT; the kernel then ends
// normally and leaves the context usable.
__global__ void wait_timeout_selftest_kernel(uint32_t* d_err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        pa::mbar_init(pa::smem_addr(&bar), 1);
        pa::fence_barrier_init();
    }
    __syncthreads();
    if (!pa::mbar_wait_warp(pa::smem_addr(&bar), 0) && threadIdx.x == 0)
        pa::report(d_err, PA_DERR_TIMEOUT);
}
}  // namespace

extern "C" pa_status pa_selftest_wait_timeout(uint32_t* d_err, pa_stream_t stream) {
    if (d_err == nullptr) return PA_ERR_INVALID_ARG;
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d_err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
