// dg_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "dg.h"

namespace dg {

// Kernel entry points of the dense CUDA-core family, by (op, tokens in the
// launch's chunk, rows per warp).  nullptr when that combination is not built.
const void* dense_kernel_gemv(int mt, int R, bool ksplit);
const void* dense_kernel_gateup(int mt, int R, bool ksplit);
const void* dense_kernel_head(int mt, int R, bool ksplit);
// Bulk-staged variant of the same family (dg_cc_bulk.cuh), by tokens in the chunk.
const void* bulk_kernel_gemv(int mt);
const void* bulk_kernel_gateup(int mt);
const void* bulk_kernel_head(int mt);

// MoE kernels by the most (token, slot) pairs one pass handles (1, 2, 4 or 8).
const void* moe_w1_kernel(int mtmax);
const void* moe_w2_kernel(int mtmax);
// The row-range MoE kernel (one contiguous row range of every active expert per CTA)
// and its dynamic shared memory for rpc output rows per CTA (W2; 0 for W1).
const void* moe_range_kernel_fn(bool w1, int mtmax);
size_t moe_range_smem(bool w1, int M, int topk, int K, int rpc);

// tcgen05 family (dg_tc_dense.cu): padded token count, fixed K-split of a shape,
// workspace bytes, and the launcher (bf16 linear or interleaved gate/up rows).
struct DeviceInfo;
int tc_mp(int M);
int tc_nsplit(const DeviceInfo* dev, int N, int K, int M, bool fixed);
// Queries (once per device, from dg_init) how many thread-block clusters of each size
// the tensor-core kernels can keep resident, so that no launch -- inside a stream
// capture or not -- queries the driver for its K-split.
void tc_capacity_init(const DeviceInfo* dev);
size_t tc_workspace_bytes(int M, int N, int K);

dg_status launch_tc(bool gate_up, const DeviceInfo* dev, const dg_choice& c, const void* x, const void* W,
                    void* out, int M, int N, int K, int ld_out, void* ws, size_t ws_bytes, cudaStream_t stream);

// Warp-level tensor-core family (dg_mma_dense.cu): bf16 linear (gate_up = false) or
// interleaved gate/up rows, 1..16 token rows.
dg_status launch_mw(bool gate_up, const DeviceInfo* dev, const dg_choice& c, const void* x, const void* W, void* out,
                    int M, int N, int K, int ld_out, cudaStream_t stream);

// A8W8 block-scaled linear on the tcgen05 family (dg_tc_dense.cu): the fixed K-split
// of a shape and the launcher; the activation quantisation alone (dg_a8.cu).
constexpr int kA8MaxRows = 64;
int tc_a8_nsplit(const DeviceInfo* dev, int N, int K);
size_t a8_workspace_bytes(int M, int K);
dg_status launch_tc_a8(const DeviceInfo* dev, const dg_choice& c, const void* x, const void* Wq, const float* sw,
                       void* y, int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t stream);
dg_status launch_a8_quant(const void* x, void* q, float* sx, int M, int K, cudaStream_t stream);

// tcgen05 fp8 head (dg_tc_head.cu): shared memory for (K, stages) and the launcher.
size_t tc_head_smem(int K, int stages);
dg_status launch_tc_head(const DeviceInfo* dev, const dg_choice& c, const void* x, const void* Wq,
                         const float* scale, void* logits, int32_t* argmax, int M, int N, int K, void* ws,
                         size_t ws_bytes, cudaStream_t stream);
// tcgen05 MoE W1 / W2 (dg_tc_moe.cu).
struct MoeArgs;
dg_status launch_tc_moe(bool w1, const DeviceInfo* dev, const dg_choice& c, const MoeArgs& m, cudaStream_t stream);

// Smallest row bucket the fp8 head sends to the tensor cores, and the largest K
// whose split activations fit in shared memory.
constexpr int kTcHeadMinRows = 2;
// Smallest row buckets the MoE calls send to the tensor cores, and the largest that
// take the CUDA-core row-range order (measured on GB300 with graphs of 16 calls over
// 8 routings: the row-range W2 beats the tensor cores up to 4 token rows, 35.3 vs
// 38.0 us at 4; the tensor cores win from 6 rows up, the (expert, N-tile) order
// takes W1 at 3-6 rows).
constexpr int kTcMoeW1MinRows = 8;
constexpr int kTcMoeW2MinRows = 5;
constexpr int kMoeRangeMaxRowsW1 = 2;
constexpr int kMoeRangeMaxRowsW2 = 4;
// Work order of the CUDA-core MoE kernels (choice params[5]): (expert, N-tile) units
// walked by persistent CTAs, or one contiguous row range of every expert per CTA.
constexpr int kMoeOrderUnits = 1;
constexpr int kMoeOrderRange = 2;
constexpr int kTcHeadMaxK = 8192;

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;
    int driver_version = 0, runtime_version = 0;
    char name[256] = {0};
};

// Properties of the current device (initialising it on first use); nullptr on failure.
const DeviceInfo* current_device(dg_status* err);

// Resident CTAs per SM for `fn` with `threads` threads and `smem` dynamic bytes
// (cached); also raises the kernel's dynamic shared memory limit once.
int occupancy(const void* fn, int threads, size_t smem);

// Launch with this library's attributes (programmatic dependent launch when enabled).
bool pdl_enabled();
cudaError_t launch_kernel(const void* fn, unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                          void** args);
// The same as a cooperative launch: the runtime starts it only with every CTA resident
// at once, whatever else the GPU runs -- for kernels with a grid-wide barrier.
cudaError_t launch_kernel_cooperative(const void* fn, unsigned grid, unsigned block, size_t smem,
                                      cudaStream_t stream, void** args);

// While an instance lives, launch_kernel on this thread checks nothing more and
// launches nothing (returns success): an entry point run under it performs every
// argument, shape, variant and workspace check of a real call -- the same code --
// and queues no work.
struct CheckOnly {
    CheckOnly();
    ~CheckOnly();
    CheckOnly(const CheckOnly&) = delete;
    CheckOnly& operator=(const CheckOnly&) = delete;
};

// Upper bound on the grid of any persistent launch of the head, and the bytes of its
// per-CTA (value, index) partials for 8 rows beyond the workspace header -- the one
// constant the workspace size and the no-allocation scratch are both built from.
constexpr int kMaxGrid = 4096;
constexpr size_t kHeadPartialBytes = static_cast<size_t>(kMaxGrid) * 8 * 8;

// Maximum dynamic shared memory any launch of this library asks for.
constexpr size_t kMaxDynSmem = 200 * 1024;
// Budget for staged activations of the dense CUDA-core family.
constexpr size_t kXsBudget = 96 * 1024;

// Row buckets of the bf16 linear and gate/up (measured on GB300, graph replay over
// weights beyond L2): the CUDA cores below kMwMinRows*, the warp-level tensor cores
// (mma.sync) up to kMwMaxRows*, the tcgen05 tiles above (always from the 16-row bucket).
constexpr int kMwMinRowsLinear = 2;
constexpr int kMwMinRowsGateUp = 3;
constexpr int kMwMaxRowsLinear = 12;
constexpr int kMwMaxRowsGateUp = 8;
constexpr int kTcMinRows = 13;
// Most token rows of one bf16 linear or gate/up call (the mid-M buckets 129..512 run
// on the tensor cores in chunks of up to 256 tokens).
constexpr int kMaxDenseRows = 512;

// Compiled default choice for (op, M, N, K).
void default_choice(dg_op op, int M, int N, int K, dg_choice* out);

// Build identity string for tables.
const char* build_id();

}  // namespace dg
