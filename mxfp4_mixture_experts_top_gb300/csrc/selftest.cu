// Self-test of the bounded pipeline wait (ptx::mbar_wait), the routine every
// wait of the GEMM pipelines goes through: one thread waits on a shared-memory
// mbarrier that nothing arrives on, so the wait can only end by running out
// its time limit or by the CTA's abort flag, which a second warp may set. The
// kernel records MOE_ERR_TIMEOUT in the error word, like a pipeline that gave
// up, and returns: no fault, no trap, the context stays usable.
#include <cstdint>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_kernel(uint64_t limit_ns, uint64_t abort_after_ns, int32_t *err, uint64_t *elapsed)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    __shared__ uint64_t t_start;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
        t_start = ptx::globaltimer_ns();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns);
        *elapsed = ptx::globaltimer_ns() - t0;
        if (!ok) atomicCAS(err, 0, DEV_ERR_TIMEOUT);
    } else if (threadIdx.x == 32 && abort_after_ns > 0) {
        // ends: abort_after_ns < limit_ns <= 1 s (checked on the host)
        while (ptx::globaltimer_ns() - t_start < abort_after_ns) __nanosleep(1000);
        abort_flag = 1;
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(uint64_t limit_ns, uint64_t abort_after_ns, int32_t *d_error_word,
                                                  uint64_t *d_elapsed_ns, void *stream)
{
    if (limit_ns == 0 || limit_ns > 1000000000ull || abort_after_ns >= limit_ns) return MOE_ERR_INVALID_ARG;
    if (!d_error_word || !d_elapsed_ns) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_error_word) & 3u) || (reinterpret_cast<uintptr_t>(d_elapsed_ns) & 7u))
        return MOE_ERR_MISALIGNED;
    moe::bounded_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, abort_after_ns, d_error_word,
                                                                            d_elapsed_ns);
    moe::note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
