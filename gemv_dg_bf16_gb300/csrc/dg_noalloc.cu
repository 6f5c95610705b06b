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
// kMaxGrid CTAs x 8 rows: built from the same constants as
// dg_workspace_bytes(DG_OP_HEAD_FP8_ARGMAX, ...), which the head checks its workspace against.
constexpr size_t kNoAllocBytes = dg::kWsData + dg::kHeadPartialBytes;
static_assert(kNoAllocBytes % 256 == 0, "the scratch keeps the workspace's 256-byte granularity");

__device__ __align__(256) uint8_t g_head_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_addr[64];

// The array's device address on the current device, looked up once per device.
dg_status scratch_address(void** out)
{
    dg_status s;
    const dg::DeviceInfo* dev = dg::current_device(&s);
    if (!dev) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev->device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DG_ERR_CUDA;
        }
        g_scratch_addr[dev->device] = p;
    }
    *out = g_scratch_addr[dev->device];
    return DG_OK;
}

}  // namespace

extern "C" dg_status dg_head_fp8_argmax_noalloc(const void* x, const void* Wq, const float* scale,
                                               void* logits, int32_t* argmax, int M, int N, int K,
                                               dg_stream_t stream, const dg_choice* choice)
{
    void* ws = nullptr;
    dg_status s = scratch_address(&ws);
    if (s != DG_OK) return s;
    // Every check of the call first -- the workspace entry point's own code, run with
    // its launch suppressed -- so that a refused call queues nothing on the stream.
    {
        dg::CheckOnly check;
        s = dg_head_fp8_argmax(x, Wq, scale, logits, argmax, M, N, K, ws, kNoAllocBytes, stream, choice);
    }
    if (s != DG_OK) {
        if (s == DG_ERR_WORKSPACE_TOO_SMALL)
            std::fprintf(stderr, "libdecodegemm: dg_head_fp8_argmax_noalloc: this launch needs more than the "
                         "%d CTA partial slots of its static scratch (use fewer, larger CTAs)\n", dg::kMaxGrid);
        return s;
    }
    // The status word and the ticket must start at zero; the partials are written
    // before they are read.  A memset node allocates nothing.
    if (cudaMemsetAsync(ws, 0, dg::kWsData, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return dg_head_fp8_argmax(x, Wq, scale, logits, argmax, M, N, K, ws, kNoAllocBytes, stream, choice);
}

extern "C" dg_status dg_head_fp8_argmax_noalloc_status(int32_t* host_out, dg_stream_t stream)
{
    if (!host_out) return DG_ERR_INVALID_ARG;
    void* ws = nullptr;
    dg_status s = scratch_address(&ws);
    if (s != DG_OK) return s;
    return dg_device_status(ws, host_out, stream);
}

extern "C" dg_status dg_head_fp8_argmax_noalloc_scratch(void** device_ptr)
{
    if (!device_ptr) return DG_ERR_INVALID_ARG;
    return scratch_address(device_ptr);
}
