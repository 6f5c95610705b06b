// dg_selftest.cu -- test hooks of the library:
//  * a health check of the bounded-wait mechanism every pipelined kernel relies
//    on: one CTA waits on an mbarrier that nothing ever completes, gives up after
//    `timeout_us`, and reports DG_DEVERR_WAIT_TIMEOUT through the workspace status
//    word, leaving the context usable;
//  * an export of the MoE routing tables, computed by the same routing scan the
//    MoE kernels run, so that they can be compared bit for bit with the oracle.
#include "dg_internal.h"
#include "dg_moe.cuh"
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

// ------------------------------------------------------------------ routing export

namespace dg {
namespace {

// One CTA runs the MoE kernels' routing scan and writes its tables out.
__global__ void route_debug_kernel(const int32_t* ids, int M, int topk, int E, int32_t* out, uint8_t* ws)
{
    __shared__ Route R;
    route_scan(R, ids, M, topk, E, ws);
    int32_t* o_valid = out + 2;
    int32_t* o_nvalid = o_valid + kMoeMaxPairs;
    int32_t* o_experts = o_nvalid + 16;
    int32_t* o_offs = o_experts + kMoeMaxPairs;
    int32_t* o_ptok = o_offs + kMoeMaxPairs + 1;
    int32_t* o_pslot = o_ptok + kMoeMaxPairs;
    if (threadIdx.x == 0) {
        out[0] = R.U;
        out[1] = R.P;
    }
    for (int i = threadIdx.x; i < kMoeMaxPairs; i += blockDim.x) {
        const bool in_pairs = i < M * topk;
        o_valid[i] = in_pairs ? R.valid[i] : 0;
        o_experts[i] = i < R.U ? R.experts[i] : -1;
        o_ptok[i] = i < R.P ? R.ptok[i] : -1;
        o_pslot[i] = i < R.P ? R.pslot[i] : -1;
    }
    for (int i = threadIdx.x; i <= kMoeMaxPairs; i += blockDim.x) o_offs[i] = i <= R.U ? R.offs[i] : -1;
    for (int t = threadIdx.x; t < 16; t += blockDim.x) o_nvalid[t] = t < M ? R.nvalid[t] : 0;
}

}  // namespace
}  // namespace dg

extern "C" dg_status dg_moe_route_debug(const int32_t* topk_ids, int M, int topk, int E, int32_t* out, void* ws,
                                        dg_stream_t stream)
{
    if (!topk_ids || !out || !ws) return DG_ERR_INVALID_ARG;
    if (M < 1 || M > 16 || topk < 1 || topk > 8 || E < 1 || E > dg::kMoeMaxE) return DG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 15u) return DG_ERR_ALIGNMENT;
    dg_status s;
    if (!dg::current_device(&s)) return s;
    dg::route_debug_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(topk_ids, M, topk, E, out,
                                                                                  static_cast<uint8_t*>(ws));
    if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
    return DG_OK;
}
