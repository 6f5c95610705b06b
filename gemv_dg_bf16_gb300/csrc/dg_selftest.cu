// dg_selftest.cu -- health check of the bounded-wait mechanism every pipelined
// kernel of this library relies on: one CTA waits on an mbarrier that nothing
// ever completes, gives up after `timeout_us`, and reports DG_DEVERR_WAIT_TIMEOUT
// through the workspace status word, leaving the context usable.
#include "dg_internal.h"
#include "dg_tc_common.cuh"

namespace dg {
namespace {

__global__ void wait_timeout_kernel(uint8_t* ws, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::bar_init(tc::su32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Phase 0 never completes: no thread arrives and no copy is in flight.
        if (!tc::bar_wait_for(tc::su32(&bar), 0u, &abort_flag, timeout_ns)) set_status(ws, DG_DEVERR_WAIT_TIMEOUT);
    }
}

}  // namespace
}  // namespace dg

extern "C" dg_status dg_selftest_wait_timeout(void* ws, int timeout_us, dg_stream_t stream)
{
    if (!ws || timeout_us < 1 || timeout_us > 2000000) return DG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 15u) return DG_ERR_ALIGNMENT;
    dg_status s;
    if (!dg::current_device(&s)) return s;
    dg::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint8_t*>(ws), static_cast<unsigned long long>(timeout_us) * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
    return DG_OK;
}
