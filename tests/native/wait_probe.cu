// Test-only probe of the library's bounded mbarrier wait (pa::tc::mbar_wait)
// and its device status word.  One CTA of one warp waits on an mbarrier; with
// arrive == 0 nothing ever arrives, so the wait must give up after `limit`
// SM cycles, set PA_DEVICE_TIMEOUT_MMA in the library's status word (the
// address the library's own kernels use) and return.  Nothing else is in
// flight: no cluster, no TMA, no tensor-core work.  Nothing in the library
// uses this file.
#include <cstdint>

#include "pa_internal.h"
#include "sm103_tc.cuh"

namespace {

__global__ void wait_probe_kernel(int32_t *status, long long limit, int arrive, int32_t *result) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        pa::tc::mbar_init(&bar, 1);
        pa::tc::fence_mbar_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) pa::tc::mbar_arrive(&bar);    // completes phase 0
    __syncwarp();
    const long long t0 = clock64();
    const bool ok = pa::tc::mbar_wait(&bar, 0, limit);
    const long long waited = clock64() - t0;
    if (!ok && threadIdx.x == 0) atomicCAS(status, 0, PA_DEVICE_TIMEOUT_MMA);
    if (threadIdx.x == 0) {
        result[0] = ok ? 1 : 2;
        result[1] = (int32_t)(waited > 0x7fffffffll ? 0x7fffffffll : waited);
    }
}

}  // namespace

// Launch the probe on the current device and wait for it.  Returns 0 and fills
// out[0] (1: the wait succeeded, 2: it gave up) and out[1] (cycles spent
// waiting), or a negative value when a CUDA call failed.
extern "C" int probe_wait(long long limit, int arrive, int32_t *out) {
    int32_t *status = pa::device_status_ptr();
    if (!status) return -1;
    int32_t *result = nullptr;
    if (cudaMalloc(&result, 2 * sizeof(int32_t)) != cudaSuccess) return -2;
    wait_probe_kernel<<<1, 32>>>(status, limit, arrive, result);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(out, result, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost);
    cudaFree(result);
    return e == cudaSuccess ? 0 : -3;
}
