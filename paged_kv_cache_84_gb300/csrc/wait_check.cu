// A check of the bounded waits' give-up path on the GPU.
//
// Every mbarrier wait of the attention kernels gives up after a time limit,
// sets PKV_DEVERR_TIMEOUT and reports failure, and the kernels then leave
// in order: the failure becomes CTA-uniform through shared memory before
// any later barrier, and the tensor-memory owner frees its columns.  This
// kernel has the same skeleton on a small scale — warp 1 owns tensor memory
// and waits for nothing, warp 0 stands for a producer waiting for a free
// stage, warps 2 and 3 for consumers waiting for data — and its barriers
// are never arrived at, so every wait runs out after `limit_ns`.  It runs
// the same wait routine as the attention kernels (mbar_wait), with a short
// limit instead of their 2 s.  Nothing here breaks an attention kernel: the
// waits time out because nothing is ever meant to arrive.
#include "pkv.h"
#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

constexpr int kCheckThreads = 128;

__global__ void __launch_bounds__(kCheckThreads, 1) wait_check_kernel(uint32_t *err, uint32_t *report,
                                                                        uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t gave_up;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        gave_up = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;
    if (warp == 0) {                                 // a producer: one lane waits for a free stage
        if (lane == 0) ok = mbar_wait(smem_u32(&bars[0]), 0, err, limit_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    } else if (warp >= 2) {                          // consumers: every lane waits for data
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[1]), 0, err, limit_ns));
    }
    if (!ok && lane == 0) atomicOr(&gave_up, 1u << warp);
    tc_fence_before();
    __syncthreads();                                 // every warp reaches it, failed or not
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
    if (threadIdx.x == 0) {
        report[0] = gave_up;                         // one bit per warp whose wait gave up
        report[1] = (uint32_t)((globaltimer_ns() - t0) / 1000u);   // microseconds in the kernel
    }
}

}  // namespace pkv

extern "C" pkv_status pkv_check_bounded_wait(uint32_t *device_error, uint32_t *report, uint32_t limit_us,
                                             cudaStream_t stream)
{
    if (!device_error || !report || limit_us == 0 || limit_us > 100000u) return PKV_ERR_INVALID_ARG;
    pkv::wait_check_kernel<<<1, pkv::kCheckThreads, 0, stream>>>(device_error, report,
                                                                 (uint64_t)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
