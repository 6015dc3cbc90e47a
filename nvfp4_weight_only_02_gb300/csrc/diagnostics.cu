// diagnostics.cu -- self-checks of the bounded-wait machinery.  Each kernel
// waits for something that never happens; the wait must give up after its
// limit, record NVFP4_ERR_TIMEOUT in the status word and return, leaving the
// CUDA context usable.  Nothing here faults, traps or hangs.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace nvfp4 {

// An mbarrier that expects one arrival which never comes.
__global__ void wait_mbarrier_kernel(uint32_t *ctl)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0))
        record_status(ctl, NVFP4_ERR_TIMEOUT);
}

// A kernel that has counted arrivals at a few output tiles (as a decode GEMM
// block does before its last-arriver test) and then gives up on a wait: it
// leaves the counters non-zero and marks the workspace.
__global__ void wait_tiles_kernel(uint32_t *ctl)
{
    __shared__ uint64_t bar;
    uint32_t *tcnt = ctl + kCtlBytes / 4;
    if (threadIdx.x < 4)
        atomicAdd(&tcnt[threadIdx.x * 7], 1u);
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0))
        record_timeout_tiles(ctl);
}

// A grid barrier told to expect one block more than were launched.
__global__ void wait_grid_kernel(uint32_t *ctl, uint32_t expected)
{
    grid_barrier(ctl, expected);
}

cudaError_t launch_wait_selftest(uint32_t *ctl, int which, cudaStream_t s)
{
    if (which == 0) {
        wait_mbarrier_kernel<<<1, 32, 0, s>>>(ctl);
        return cudaGetLastError();
    }
    if (which == 2) {
        wait_tiles_kernel<<<1, 32, 0, s>>>(ctl);
        return cudaGetLastError();
    }
    uint32_t *c = ctl;
    uint32_t expected = 3;
    void *args[] = {&c, &expected};
    cudaError_t e = cudaLaunchCooperativeKernel((const void *)wait_grid_kernel, dim3(2), dim3(32), args, 0, s);
    if (e != cudaSuccess)
        return e;
    // the blocks that gave up left their arrivals counted: clear them
    return cudaMemsetAsync(ctl + CTL_BAR_COUNT, 0, 4, s);
}

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_wait_selftest(void *workspace, int which, void *stream)
{
    if (!workspace || which < 0 || which > 2)
        return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st;
    if (!nvfp4::device_info(&st))
        return st;
    return nvfp4::launch_wait_selftest((uint32_t *)workspace, which, (cudaStream_t)stream) == cudaSuccess
               ? NVFP4_OK
               : NVFP4_ERR_CUDA;
}
