// dg_api.cu -- the libdecodegemm C ABI: argument checks, kernel choice, launch.
//
// Nothing here allocates device memory or synchronises the host with a stream
// (dg_device_status excepted, which exists for tests and health checks).
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "dg_cc_bulk.cuh"
#include "dg_cc_dense.cuh"
#include "dg_internal.h"
#include "dg_moe.cuh"

namespace dg {

namespace {

std::mutex g_mu;
DeviceInfo g_dev[64];
bool g_dev_ok[64];
// Both per device: a kernel's attributes and occupancy belong to the device it runs on.
std::map<std::tuple<int, const void*, int, size_t>, int> g_occ;
std::map<std::pair<int, const void*>, bool> g_attr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

const DeviceInfo* current_device(dg_status* err)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        if (err) *err = DG_ERR_NO_DEVICE;
        return nullptr;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev_ok[dev]) return &g_dev[dev];
    }
    dg_status s = dg_init(dev);
    if (s != DG_OK) {
        if (err) *err = s;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    return &g_dev[dev];
}

namespace {
std::atomic<int> g_launch_flags{DG_LAUNCH_PDL};
}

bool pdl_enabled() { return (g_launch_flags.load(std::memory_order_relaxed) & DG_LAUNCH_PDL) != 0; }

namespace {
thread_local int t_check_only = 0;
}

CheckOnly::CheckOnly() { ++t_check_only; }
CheckOnly::~CheckOnly() { --t_check_only; }

cudaError_t launch_kernel(const void* fn, unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                          void** args)
{
    if (t_check_only) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_kernel_cooperative(const void* fn, unsigned grid, unsigned block, size_t smem,
                                      cudaStream_t stream, void** args)
{
    if (t_check_only) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int occupancy(const void* fn, int threads, size_t smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        dev = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_attr[std::make_pair(dev, fn)]) {
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxDynSmem));
        g_attr[std::make_pair(dev, fn)] = true;
    }
    auto key = std::make_tuple(dev, fn, threads, smem);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    g_occ[key] = n;
    return n;
}

void default_choice(dg_op op, int M, int N, int K, dg_choice* out)
{
    std::memset(out, 0, sizeof *out);
    out->variant = DG_VAR_CC_WARP;
    switch (op) {
    case DG_OP_GEMV_BF16:
    case DG_OP_GATE_UP_SILU: {
        const bool lin = op == DG_OP_GEMV_BF16;
        if (M >= kTcMinRows || M > (lin ? kMwMaxRowsLinear : kMwMaxRowsGateUp)) {
            out->variant = DG_VAR_TC;      // a real dense contraction: tcgen05 tiles
            break;
        }
        if (M >= (lin ? kMwMinRowsLinear : kMwMinRowsGateUp)) {
            out->variant = DG_VAR_MMA;     // warp-level tensor cores, geometry derived at launch
            break;
        }
        // Rows per warp [0], warps per CTA [1] and K-split warps [3] as dg_sweep
        // measured them on GB300 for one and two tokens: long rows with few row groups
        // share each group's K segments between warps; many short rows do not.
        const long rows = op == DG_OP_GATE_UP_SILU ? 2L * N : static_cast<long>(N);
        const int nseg = (K + kSeg - 1) / kSeg;
        int R, wpc, ks;
        if (op == DG_OP_GATE_UP_SILU) {
            R = 2;
            wpc = M <= 1 ? 4 : 8;
            ks = M <= 1 ? 4 : 1;
        } else if (rows >= 32768) {
            R = M <= 1 ? 1 : 2;
            wpc = 8;
            ks = 1;
        } else if (rows >= 12288) {
            R = 4;
            wpc = 4;
            ks = M <= 1 ? 4 : 2;
        } else if (rows >= 8192) {
            R = 2;
            wpc = M <= 1 ? 4 : 8;
            ks = 1;
        } else {
            R = (M <= 1 && K <= 4096) ? 2 : 4;
            wpc = 8;
            ks = 2;
        }
        while (ks > 1 && nseg < ks) ks /= 2;          // no warp without a segment
        out->params[0] = R;
        out->params[1] = wpc;
        out->params[3] = ks > 1 ? ks : 0;
        break;
    }
    case DG_OP_HEAD_FP8_ARGMAX:
        if (M >= kTcHeadMinRows && K <= kTcHeadMaxK) {
            out->variant = DG_VAR_TC;      // fp8 MMA on split activations
            break;
        }
        // measured on GB300 (dg_sweep over the 248320 x 4096 head)
        out->params[0] = M == 4 ? 4 : (M <= 3 ? 8 : 4);
        out->params[1] = M <= 4 ? 4 : 8;
        break;
    // MoE: [1] warps per CTA, [3] N-tile (W1: gate/up columns, W2: output rows),
    // [4] pairs per pass -- the GB300 dg_sweep picks per row bucket.
    case DG_OP_MOE_W1:
        if (M >= kTcMoeW1MinRows) {
            out->variant = DG_VAR_TC;
            break;
        }
        if (M <= kMoeRangeMaxRowsW1) {         // one row range of every expert per CTA
            out->params[0] = 4;
            out->params[1] = 4;
            out->params[4] = 2;
            out->params[5] = kMoeOrderRange;
            break;
        }
        out->params[0] = 4;
        out->params[1] = 8;
        out->params[3] = M <= 1 ? 32 : (M <= 2 ? 64 : 0);
        out->params[4] = M <= 2 ? 4 : 2;
        break;
    case DG_OP_MOE_W2:
        if (M >= kTcMoeW2MinRows) {
            out->variant = DG_VAR_TC;
            break;
        }
        if (M <= kMoeRangeMaxRowsW2) {
            out->params[0] = 4;
            out->params[1] = 8;
            out->params[4] = 2;
            out->params[5] = kMoeOrderRange;
            break;
        }
        out->params[0] = 4;
        out->params[1] = M <= 2 ? 8 : 4;
        out->params[3] = M <= 1 ? 64 : (M <= 2 ? 128 : (M <= 4 ? 0 : 64));
        out->params[4] = M <= 1 ? 1 : 2;
        break;
    case DG_OP_GEMV_A8W8:
        out->variant = DG_VAR_TC;          // fp8 MMA on the quantised activations
        // Measured on GB300 (32768x1024, 8192x4096): the fused quantisation ties with a
        // quantisation launch of its own up to 16 rows; beyond, every CTA re-quantising
        // all rows costs more than one extra launch (12.7 -> 9.7 us at 32 rows).
        out->params[1] = M > 16 ? 1 : 0;
        break;
    default:
        break;
    }
}

#ifndef DG_BUILD_ID
#define DG_BUILD_ID "dev"
#endif

const char* build_id() { return DG_BUILD_ID; }

}  // namespace dg

using namespace dg;

extern "C" {

dg_status dg_init(int device)
{
    if (device < 0 || device >= 64) return DG_ERR_INVALID_ARG;
    if (cudaSetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_NO_DEVICE;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_NO_DEVICE;
    }
    if (prop.major != 10 || prop.minor != 3) {
        std::fprintf(stderr, "libdecodegemm: device %d is sm_%d%d; this build runs on sm_103 only\n",
                     device, prop.major, prop.minor);
        return DG_ERR_NO_DEVICE;
    }
    DeviceInfo info;
    info.device = device;
    info.sm_count = prop.multiProcessorCount;
    info.cc_major = prop.major;
    info.cc_minor = prop.minor;
    info.max_smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
    cudaDriverGetVersion(&info.driver_version);
    cudaRuntimeGetVersion(&info.runtime_version);
    std::snprintf(info.name, sizeof info.name, "%s", prop.name);
    bool first = false;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        first = !g_dev_ok[device];
        g_dev[device] = info;
        g_dev_ok[device] = true;
    }
    if (first) {
        tc_capacity_init(&info);
        const char* path = std::getenv("DG_TABLE");
        if (path && *path) dg_table_load(path);   // refusal prints one line; defaults stay
    }
    return DG_OK;
}

const char* dg_status_str(dg_status s)
{
    switch (s) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument";
    case DG_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case DG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case DG_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DG_ERR_CUDA: return "CUDA error";
    case DG_ERR_TABLE_REFUSED: return "shape table refused";
    case DG_ERR_NO_DEVICE: return "no usable sm_103 device";
    case DG_ERR_BAD_VARIANT: return "bad kernel variant";
    default: return "unknown status";
    }
}

size_t dg_workspace_bytes(dg_op op, int M, int N, int K, int topk)
{
    (void)K;
    size_t b = kWsData;
    switch (op) {
    case DG_OP_GEMV_BF16:
        if (M > 0 && N > 0 && K > 0) b = tc_workspace_bytes(M, N, K);
        break;
    case DG_OP_GATE_UP_SILU:
        if (M > 0 && N > 0 && K > 0) b = tc_workspace_bytes(M, 2 * N, K);
        break;
    case DG_OP_HEAD_FP8_ARGMAX:
        b += kHeadPartialBytes;
        break;
    case DG_OP_MOE_W2:
        if (M > 0 && topk > 0 && N > 0) b += moe_terms_bytes(M, topk, N);
        break;
    case DG_OP_GEMV_A8W8:
        if (M > 0 && K > 0) b = a8_workspace_bytes(M, K);
        break;
    default:
        break;
    }
    return b;
}

dg_status dg_device_status(const void* ws, int32_t* host_out, dg_stream_t stream)
{
    if (!ws || !host_out) return DG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_out, static_cast<const uint8_t*>(ws) + kWsStatus, sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

dg_status dg_set_launch_flags(unsigned flags)
{
    if (flags & ~static_cast<unsigned>(DG_LAUNCH_PDL)) return DG_ERR_INVALID_ARG;
    g_launch_flags.store(static_cast<int>(flags));
    return DG_OK;
}

unsigned dg_launch_flags(void) { return static_cast<unsigned>(g_launch_flags.load()); }

dg_status dg_device_status_clear(void* ws, dg_stream_t stream)
{
    if (!ws) return DG_ERR_INVALID_ARG;
    if (cudaMemsetAsync(static_cast<uint8_t*>(ws) + kWsStatus, 0, sizeof(int32_t),
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // extern "C"

namespace dg {
namespace {

dg_status resolve_choice(dg_op op, int M, int N, int K, const dg_choice* in, dg_choice* out)
{
    if (in && in->variant != DG_VAR_DEFAULT) {
        *out = *in;
        return DG_OK;
    }
    return dg_select(op, M, N, K, out);
}

// Bulk-staged variant: one (or two) persistent CTAs per SM, a deep shared-memory ring.
dg_status launch_bulk(dg_op op, const DeviceInfo* dev, const dg_choice& c, DenseArgs a, int M, size_t ws_bytes,
                      cudaStream_t stream)
{
    const int esz = (op == DG_OP_HEAD_FP8_ARGMAX) ? 1 : 2;
    const int rw = (op == DG_OP_GATE_UP_SILU) ? 2 : 1;
    const int cps = c.params[2] > 0 ? c.params[2] : 1;
    if (c.params[0] != 0 || c.params[1] < 0 || c.params[1] > 32 || c.params[1] == 1 || cps > 2)
        return DG_ERR_BAD_VARIANT;
    int mt_max = static_cast<int>(kXsBudget / (static_cast<size_t>(a.K) * 2));
    if (mt_max > 8) mt_max = 8;
    if (mt_max < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (op == DG_OP_HEAD_FP8_ARGMAX && M > mt_max) return DG_ERR_UNSUPPORTED_SHAPE;
    const size_t stage = static_cast<size_t>(kBulkConsumers) * rw * kSeg * esz;
    const size_t budget = (cps == 1 ? kMaxDynSmem : kMaxDynSmem / 2 - 8 * 1024);
    for (int t0 = 0; t0 < M; t0 += mt_max) {
        const int mt = (M - t0 < mt_max) ? M - t0 : mt_max;
        const void* fn = op == DG_OP_GEMV_BF16      ? bulk_kernel_gemv(mt)
                         : op == DG_OP_GATE_UP_SILU ? bulk_kernel_gateup(mt)
                                                    : bulk_kernel_head(mt);
        if (!fn) return DG_ERR_BAD_VARIANT;
        const size_t xbytes = (static_cast<size_t>(mt) * a.K * 2 + 127) / 128 * 128;
        if (xbytes + 2 * stage + 64 > budget) return DG_ERR_UNSUPPORTED_SHAPE;
        int stages = c.params[1];
        const int fit = static_cast<int>((budget - xbytes - 64) / (stage + 16));
        if (stages == 0) stages = fit < 32 ? fit : 32;
        if (stages < 2 || stages > fit) return DG_ERR_BAD_VARIANT;
        const size_t smem = xbytes + static_cast<size_t>(stages) * (stage + 16);
        const int occ = occupancy(fn, kBulkThreads, smem);
        if (occ < 1) return DG_ERR_UNSUPPORTED_SHAPE;
        const long long grid = static_cast<long long>(dev->sm_count) * (occ < cps ? occ : cps);
        if (op == DG_OP_HEAD_FP8_ARGMAX && ws_bytes < kWsData + static_cast<size_t>(grid) * cpow2(mt) * 8)
            return DG_ERR_WORKSPACE_TOO_SMALL;
        DenseArgs la = a;
        la.t0 = t0;
        void* args[] = {&la, &stages};
        if (launch_kernel(fn, static_cast<unsigned>(grid), kBulkThreads, smem, stream, args) !=
            cudaSuccess) {
            cudaGetLastError();
            return DG_ERR_CUDA;
        }
    }
    return DG_OK;
}

// Launch the dense CUDA-core family over token chunks.
dg_status launch_dense(dg_op op, const DeviceInfo* dev, const dg_choice& c, DenseArgs a, int M,
                       size_t ws_bytes, cudaStream_t stream)
{
    if (c.variant == DG_VAR_CC_BULK) return launch_bulk(op, dev, c, a, M, ws_bytes, stream);
    const int esz = (op == DG_OP_HEAD_FP8_ARGMAX) ? 1 : 2;
    (void)esz;
    int R = c.params[0] > 0 ? c.params[0] : 4;
    const int wpc = c.params[1] > 0 ? c.params[1] : 8;
    const int cap = c.params[2];
    const int ks = c.params[3] > 0 ? c.params[3] : 1;
    if ((R != 1 && R != 2 && R != 4 && R != 8) || wpc < 1 || wpc > 8 || cap < 0)
        return DG_ERR_BAD_VARIANT;
    if ((ks != 1 && ks != 2 && ks != 4 && ks != 8) || wpc % ks != 0) return DG_ERR_BAD_VARIANT;
    if (op == DG_OP_GATE_UP_SILU && R < 2) return DG_ERR_BAD_VARIANT;
    int mt_max = static_cast<int>(kXsBudget / (static_cast<size_t>(a.K) * 2));
    if (mt_max > 8) mt_max = 8;
    if (mt_max < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (op == DG_OP_HEAD_FP8_ARGMAX && M > mt_max) return DG_ERR_UNSUPPORTED_SHAPE;
    for (int t0 = 0; t0 < M; t0 += mt_max) {
        const int mt = (M - t0 < mt_max) ? M - t0 : mt_max;
        int r = R;
        while (r > 1 && r * cpow2(mt) > 32) r >>= 1;       // same arithmetic, fewer rows per warp
        if (op == DG_OP_GATE_UP_SILU && r < 2) return DG_ERR_UNSUPPORTED_SHAPE;
        const int kse = mt <= 2 ? ks : 1;                 // K-split kernels exist for 1-2 token chunks
        const void* fn = op == DG_OP_GEMV_BF16      ? dense_kernel_gemv(mt, r, kse > 1)
                         : op == DG_OP_GATE_UP_SILU ? dense_kernel_gateup(mt, r, kse > 1)
                                                    : dense_kernel_head(mt, r, kse > 1);
        if (!fn) return DG_ERR_BAD_VARIANT;
        const int threads = wpc * 32;
        const int slots = wpc / kse;                      // row groups per CTA round
        size_t smem = static_cast<size_t>(mt) * a.K * 2;
        if (kse > 1)                                      // segment partials of the K-split
            smem += static_cast<size_t>(slots) * ((a.K + kSeg - 1) / kSeg) * r * cpow2(mt) * 4;
        if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;
        int occ = occupancy(fn, threads, smem);
        if (occ < 1) return DG_ERR_UNSUPPORTED_SHAPE;
        if (cap > 0 && occ > cap) occ = cap;
        DenseArgs la = a;
        la.t0 = t0;
        la.groups = (a.N + r - 1) / r;
        la.ksplit = kse;
        long long need = (la.groups + slots - 1) / slots;
        long long grid = static_cast<long long>(dev->sm_count) * occ;
        if (grid > need) grid = need;
        if (grid > kMaxGrid) grid = kMaxGrid;
        if (op == DG_OP_HEAD_FP8_ARGMAX &&
            ws_bytes < kWsData + static_cast<size_t>(grid) * cpow2(mt) * 8)
            return DG_ERR_WORKSPACE_TOO_SMALL;
        void* args[] = {&la};
        if (launch_kernel(fn, static_cast<unsigned>(grid), threads, smem, stream, args) !=
            cudaSuccess) {
            cudaGetLastError();
            return DG_ERR_CUDA;
        }
    }
    return DG_OK;
}

dg_status check_common(const void* const* ptrs, int n, void* ws, size_t ws_bytes, size_t ws_need)
{
    for (int i = 0; i < n; ++i)
        if (!ptrs[i]) return DG_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!aligned16(ptrs[i])) return DG_ERR_ALIGNMENT;
    if (!ws) return DG_ERR_INVALID_ARG;
    if (!aligned16(ws)) return DG_ERR_ALIGNMENT;
    if (ws_bytes < ws_need) return DG_ERR_WORKSPACE_TOO_SMALL;
    return DG_OK;
}

}  // namespace
}  // namespace dg

extern "C" {

dg_status dg_gemv_bf16(const void* x, const void* W, void* y, int M, int N, int K, void* ws,
                       size_t ws_bytes, dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > kMaxDenseRows || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 8 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {x, W, y};
    dg_status s = check_common(ptrs, 3, ws, ws_bytes, dg_workspace_bytes(DG_OP_GEMV_BF16, M, N, K, 0));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_GEMV_BF16, M, N, K, choice, &c)) != DG_OK) return s;
    if (c.variant == DG_VAR_TC)
        return launch_tc(false, dev, c, x, W, y, M, N, K, N, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
    if (c.variant == DG_VAR_MMA) return launch_mw(false, dev, c, x, W, y, M, N, K, N, reinterpret_cast<cudaStream_t>(stream));
    if (c.variant != DG_VAR_CC_WARP && c.variant != DG_VAR_CC_BULK) return DG_ERR_BAD_VARIANT;
    DenseArgs a{};
    a.W = static_cast<const uint8_t*>(W);
    a.x = static_cast<const uint16_t*>(x);
    a.N = N;
    a.K = K;
    a.out = static_cast<uint16_t*>(y);
    a.ld_out = N;
    a.ws = static_cast<uint8_t*>(ws);
    return launch_dense(DG_OP_GEMV_BF16, dev, c, a, M, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_gate_up_silu(const void* x, const void* W_gu, void* out, int M, int N_half, int K,
                          void* ws, size_t ws_bytes, dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > kMaxDenseRows || N_half < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 8 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {x, W_gu, out};
    dg_status s =
        check_common(ptrs, 3, ws, ws_bytes, dg_workspace_bytes(DG_OP_GATE_UP_SILU, M, N_half, K, 0));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_GATE_UP_SILU, M, N_half, K, choice, &c)) != DG_OK) return s;
    if (c.variant == DG_VAR_TC)
        return launch_tc(true, dev, c, x, W_gu, out, M, 2 * N_half, K, N_half, ws, ws_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
    if (c.variant == DG_VAR_MMA)
        return launch_mw(true, dev, c, x, W_gu, out, M, 2 * N_half, K, N_half, reinterpret_cast<cudaStream_t>(stream));
    if (c.variant != DG_VAR_CC_WARP && c.variant != DG_VAR_CC_BULK) return DG_ERR_BAD_VARIANT;
    DenseArgs a{};
    a.W = static_cast<const uint8_t*>(W_gu);
    a.x = static_cast<const uint16_t*>(x);
    a.N = 2 * N_half;
    a.K = K;
    a.out = static_cast<uint16_t*>(out);
    a.ld_out = N_half;
    a.ws = static_cast<uint8_t*>(ws);
    return launch_dense(DG_OP_GATE_UP_SILU, dev, c, a, M, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_head_fp8_argmax(const void* x, const void* Wq, const float* scale, void* logits,
                             int32_t* argmax, int M, int N, int K, void* ws, size_t ws_bytes,
                             dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > 8 || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    if (!scale || !argmax) return DG_ERR_INVALID_ARG;
    if (logits && !aligned16(logits)) return DG_ERR_ALIGNMENT;
    const void* ptrs[] = {x, Wq};
    dg_status s =
        check_common(ptrs, 2, ws, ws_bytes, dg_workspace_bytes(DG_OP_HEAD_FP8_ARGMAX, M, N, K, 0));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_HEAD_FP8_ARGMAX, M, N, K, choice, &c)) != DG_OK) return s;
    if (c.variant == DG_VAR_TC)
        return launch_tc_head(dev, c, x, Wq, scale, logits, argmax, M, N, K, ws, ws_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
    if (c.variant != DG_VAR_CC_WARP && c.variant != DG_VAR_CC_BULK) return DG_ERR_BAD_VARIANT;
    DenseArgs a{};
    a.W = static_cast<const uint8_t*>(Wq);
    a.x = static_cast<const uint16_t*>(x);
    a.N = N;
    a.K = K;
    a.out = static_cast<uint16_t*>(logits);
    a.ld_out = N;
    a.scale = scale;
    a.argmax = argmax;
    a.ws = static_cast<uint8_t*>(ws);
    return launch_dense(DG_OP_HEAD_FP8_ARGMAX, dev, c, a, M, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

// Row-range order: grid = SMs x CTAs per SM (params[2], else the occupancy limit);
// W2 cuts Nout into equal contiguous ranges (empty CTAs dropped), W1 the flattened
// (expert, column pair) list.
static dg_status launch_moe_range(bool w1, const DeviceInfo* dev, const dg_choice& c, MoeArgs a,
                                  cudaStream_t stream)
{
    const int wpc = c.params[1] > 0 ? c.params[1] : 8;
    const int mtmax = c.params[4] > 0 ? c.params[4] : 2;
    if ((c.params[0] != 0 && c.params[0] != 4) || (wpc != 4 && wpc != 8) || c.params[2] < 0 || c.params[2] > 4 ||
        c.params[3] != 0)
        return DG_ERR_BAD_VARIANT;
    const void* fn = moe_range_kernel_fn(w1, mtmax);
    if (!fn) return DG_ERR_BAD_VARIANT;
    const int threads = wpc * 32;
    const int rows = w1 ? a.I : a.Nout;
    // shared memory at the widest range any grid of >= one CTA per SM gives
    const int rpc_max = w1 ? 0 : (rows + dev->sm_count - 1) / dev->sm_count;
    size_t smem = moe_range_smem(w1, a.M, a.topk, a.K, rpc_max);
    if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;
    int occ = occupancy(fn, threads, smem);
    if (occ < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (c.params[2] > 0 && occ > c.params[2]) occ = c.params[2];
    long long grid = static_cast<long long>(dev->sm_count) * occ;
    a.tile = 0;
    if (!w1) {
        if (grid > rows) grid = rows;
        const long long rpc = (rows + grid - 1) / grid;
        grid = (rows + rpc - 1) / rpc;                      // every CTA has rows
        a.tile = static_cast<int>(rpc);
        smem = moe_range_smem(false, a.M, a.topk, a.K, a.tile);
    }
    void* args[] = {&a};
    if (launch_kernel(fn, static_cast<unsigned>(grid), threads, smem, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

static dg_status launch_moe(bool w1, const DeviceInfo* dev, const dg_choice& c, MoeArgs a,
                            cudaStream_t stream)
{
    if (c.variant == DG_VAR_TC) return launch_tc_moe(w1, dev, c, a, stream);
    if (c.variant != DG_VAR_CC_WARP) return DG_ERR_BAD_VARIANT;
    if (c.params[5] == kMoeOrderRange) return launch_moe_range(w1, dev, c, a, stream);
    if (c.params[5] != 0 && c.params[5] != kMoeOrderUnits) return DG_ERR_BAD_VARIANT;
    const int wpc = c.params[1] > 0 ? c.params[1] : 8;
    if (c.params[0] != 0 && c.params[0] != 4) return DG_ERR_BAD_VARIANT;
    if (wpc < 1 || wpc > 8 || c.params[2] < 0 || c.params[3] < 0) return DG_ERR_BAD_VARIANT;
    int tile = c.params[3];
    if (tile == 0) tile = w1 ? wpc * 2 : (wpc * 4 < 32 ? 32 : wpc * 4);
    a.tile = tile;
    if (!w1 && moe_tickets(a.M, a.Nout, tile) > kWsMaxCounters) return DG_ERR_BAD_VARIANT;
    const int mtmax = c.params[4] > 0 ? c.params[4] : 2;
    const void* fn = w1 ? moe_w1_kernel(mtmax) : moe_w2_kernel(mtmax);
    if (!fn) return DG_ERR_BAD_VARIANT;
    const int threads = wpc * 32;
    const size_t smem = static_cast<size_t>(mtmax) * a.K * 2;
    if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;
    int occ = occupancy(fn, threads, smem);
    if (occ < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (c.params[2] > 0 && occ > c.params[2]) occ = c.params[2];
    const long long grid = static_cast<long long>(dev->sm_count) * occ;
    void* args[] = {&a};
    if (launch_kernel(fn, static_cast<unsigned>(grid), threads, smem, stream, args) !=
        cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

dg_status dg_gemv_a8w8_blockscale(const void* x, const void* Wq, const float* sw, void* y, int M, int N, int K,
                                  void* ws, size_t ws_bytes, dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > kA8MaxRows || N < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {x, Wq, sw, y};
    dg_status s = check_common(ptrs, 4, ws, ws_bytes, dg_workspace_bytes(DG_OP_GEMV_A8W8, M, N, K, 0));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_GEMV_A8W8, M, N, K, choice, &c)) != DG_OK) return s;
    if (c.variant != DG_VAR_TC) return DG_ERR_BAD_VARIANT;
    return launch_tc_a8(dev, c, x, Wq, sw, y, M, N, K, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_quant_a8_blockscale(const void* x, void* q, float* sx, int M, int K, dg_stream_t stream)
{
    if (!x || !q || !sx || M < 1 || K < 1) return DG_ERR_INVALID_ARG;
    if (K % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sx)) return DG_ERR_ALIGNMENT;
    dg_status s;
    if (!current_device(&s)) return s;
    return launch_a8_quant(x, q, sx, M, K, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_moe_w1_silu(const void* x, const int32_t* topk_ids, const void* W1, const float* s1,
                         void* a_out, int M, int topk, int E, int I, int K, void* ws, size_t ws_bytes,
                         dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > 16 || topk < 1 || topk > 8 || E < 1 || E > 1024 || I < 1 || K < 1)
        return DG_ERR_INVALID_ARG;
    if (K % 16 != 0 || I % 8 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {x, topk_ids, W1, s1, a_out};
    dg_status s = check_common(ptrs, 5, ws, ws_bytes, dg_workspace_bytes(DG_OP_MOE_W1, M, I, K, topk));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_MOE_W1, M, I, K, choice, &c)) != DG_OK) return s;
    MoeArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.ids = topk_ids;
    a.W = static_cast<const uint8_t*>(W1);
    a.s = s1;
    a.out = static_cast<uint16_t*>(a_out);
    a.ws = static_cast<uint8_t*>(ws);
    a.M = M;
    a.topk = topk;
    a.E = E;
    a.I = I;
    a.K = K;
    a.Nout = 0;
    return launch_moe(true, dev, c, a, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_moe_w2(const void* a_in, const int32_t* topk_ids, const float* gw, const void* W2,
                    const float* s2, void* y, int M, int topk, int E, int I, int Nout, void* ws,
                    size_t ws_bytes, dg_stream_t stream, const dg_choice* choice)
{
    if (M < 1 || M > 16 || topk < 1 || topk > 8 || E < 1 || E > 1024 || I < 1 || Nout < 1)
        return DG_ERR_INVALID_ARG;
    if (I % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {a_in, topk_ids, gw, W2, s2, y};
    dg_status s =
        check_common(ptrs, 6, ws, ws_bytes, dg_workspace_bytes(DG_OP_MOE_W2, M, Nout, I, topk));
    if (s != DG_OK) return s;
    const DeviceInfo* dev = current_device(&s);
    if (!dev) return s;
    dg_choice c;
    if ((s = resolve_choice(DG_OP_MOE_W2, M, Nout, I, choice, &c)) != DG_OK) return s;
    MoeArgs a{};
    a.x = static_cast<const uint16_t*>(a_in);
    a.ids = topk_ids;
    a.gw = gw;
    a.W = static_cast<const uint8_t*>(W2);
    a.s = s2;
    a.out = static_cast<uint16_t*>(y);
    a.ws = static_cast<uint8_t*>(ws);
    a.M = M;
    a.topk = topk;
    a.E = E;
    a.I = I;
    a.K = I;
    a.Nout = Nout;
    return launch_moe(false, dev, c, a, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
