// dg_noalloc.cu -- dg_head_fp8_argmax_noalloc: the fp8 head + greedy pick for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the head: an engine whose memory pool is owned by someone else,
// a plugin loaded into a host that forbids device allocation, or code running
// after its memory budget has been fixed.  This entry point keeps the head's
// scratch (status word, pick ticket and per-CTA (value, index) partials) in a
// file-scope device array instead of a caller-supplied workspace.  The array is
// part of the loaded module: every GPU that loads the library holds it until
// the process exits.
#include <cstdio>
#include <mutex>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace {

// The workspace header (status word, ticket, counter region) + partials for up to
// 4096 CTAs x 8 rows: exactly
// dg_workspace_bytes(DG_OP_HEAD_FP8_ARGMAX, ...), which the head checks its workspace against.
constexpr size_t kNoAllocMaxCtas = 4096;
constexpr size_t kNoAllocBytes = dg::kWsData + kNoAllocMaxCtas * 8 * 8;

__device__ __align__(256) uint8_t g_head_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_addr[64];

// The array's device address on the current device, looked up once per device.
dg_status scratch_address(int device, void** out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DG_ERR_CUDA;
        }
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return DG_OK;
}

}  // namespace

extern "C" dg_status dg_head_fp8_argmax_noalloc(const void* x, const void* Wq, const float* scale,
                                               void* logits, int32_t* argmax, int M, int N, int K,
                                               dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > 8 || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    if (!x || !Wq || !scale || !argmax) return DG_ERR_INVALID_ARG;
    for (const void* p : {x, Wq, static_cast<const void*>(logits)})
        if (reinterpret_cast<uintptr_t>(p) & 15u) return DG_ERR_ALIGNMENT;
    dg_status s;
    const dg::DeviceInfo* dev = dg::current_device(&s);
    if (!dev) return s;
    void* ws = nullptr;
    if ((s = scratch_address(dev->device, &ws)) != DG_OK) return s;
    // The status word and the ticket must start at zero; the partials are written
    // before they are read.  A memset node allocates nothing.
    if (cudaMemsetAsync(ws, 0, dg::kWsData, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    s = dg_head_fp8_argmax(x, Wq, scale, logits, argmax, M, N, K, ws, kNoAllocBytes, stream, choice);
    if (s == DG_ERR_WORKSPACE_TOO_SMALL)
        std::fprintf(stderr, "libdecodegemm: dg_head_fp8_argmax_noalloc: this launch needs more than the "
                     "%zu CTA partial slots of its static scratch (use fewer, larger CTAs)\n", kNoAllocMaxCtas);
    return s;
}
