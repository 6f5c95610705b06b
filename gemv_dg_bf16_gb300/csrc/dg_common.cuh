// dg_common.cuh -- device helpers shared by the libdecodegemm kernels (sm_103a).
//
// The canonical reduction order (CO) every CUDA-core kernel computes:
//   K is cut into segments of kSeg = 1024 elements (the last may be short).
//   Within segment s, lane l of the warp owning a (row, token) output runs one
//   sequential fp32 fma chain, starting from +0, over the elements
//       s*kSeg + v*(32*VE) + l*VE + j     (v ascending, then j = 0..VE-1; k < K)
//   where VE is the number of weights in one 16-byte vector (8 bf16, 16 e4m3).
//   The 32 lane partials are then summed by an xor butterfly whose stages use
//   lane offsets 16, 8, 4, 2, 1 in that order (reduce_scatter below computes the
//   same tree for many outputs at once), giving p_s.  The row total is the left
//   fold ((p_0 + p_1) + p_2) + ... in fp32.
// Nothing in CO depends on rows per warp, warps per CTA, grid size, staging or
// token chunking, so every variant of the family is bitwise identical.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "dg.h"

namespace dg {

constexpr int kSeg = 1024;                 // K elements per canonical segment
constexpr unsigned kFull = 0xffffffffu;

// Workspace layout (bytes from the start of ws).  Counters live in their own
// region that no op uses for data, so one workspace may serve every op (calls
// ordered on one stream); each op leaves its counters at zero when it finishes.
constexpr size_t kWsStatus = 0;            // int32 sticky device status word
constexpr size_t kWsTicket = 16;           // uint32 ticket of single-ticket kernels (the head)
constexpr size_t kWsGridBarrier = 24;      // uint32 counter + generation of a grid barrier (tensor-core MoE W2)
constexpr size_t kWsCounters = 256;        // uint32 tickets of multi-ticket kernels (TC tiles, MoE)
constexpr size_t kWsData = 32768;          // per-op scratch data starts here
constexpr int kWsMaxCounters = static_cast<int>((kWsData - kWsCounters) / 4);

__host__ __device__ constexpr int cpow2(int v) { int p = 1; while (p < v) p <<= 1; return p; }
__host__ __device__ constexpr int clog2(int v) { int l = 0; while ((1 << l) < v) ++l; return l; }

// 16-byte streaming load of read-only weights: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte load that bypasses L1 (data written by other CTAs of this launch).
__device__ __forceinline__ uint4 ld_cg16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_cg_f32(const float* p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int ld_cg_s32(const int* p)
{
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// bf16 halves of a 32-bit word -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// acc = fma(x.lo, w.lo, acc); acc = fma(x.hi, w.hi, acc) on packed bf16 pairs, with
// the mixed-precision fma (bf16 operands, fp32 addend and result, one rounding).
__device__ __forceinline__ void fma2_bf16(float& acc, uint32_t x2, uint32_t w2)
{
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(x2), "r"(w2));
}

// Two e4m3 codes (low byte = first element) -> two fp32 values (exact), via the
// hardware e4m3x2 -> f16x2 conversion followed by f16 -> f32.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two_codes)
{
    uint32_t h2;
    const uint16_t c = static_cast<uint16_t>(two_codes & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    __half2 h;
    memcpy(&h, &h2, sizeof h);
    return __half22float2(h);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v)
{
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    uint16_t u;
    memcpy(&u, &b, sizeof u);
    return u;
}

// Reduce-scatter butterfly over the warp.  v[0..Q) are per-lane partials of Q
// independent outputs.  Stage offsets run 16, 8, 4, 2, 1; at each stage every
// lane adds its partner's value (lane ^ offset) to its own, so each output's
// sum uses the same tree as a plain xor butterfly, bit for bit.  While more
// than one output remains, a lane keeps half of them (upper half when the
// stage's lane bit is set) and sends the other half.  For Q <= 32 (a power of
// two) lane l ends with output (l >> (5 - log2 Q)) in v[0].
template <int O, int C>
struct Butterfly {
    template <int Q>
    static __device__ __forceinline__ void run(float (&v)[Q], int lane)
    {
        if constexpr (C > 1) {
            const bool up = (lane & O) != 0;
#pragma unroll
            for (int j = 0; j < C / 2; ++j) {
                const float send = up ? v[j] : v[C / 2 + j];
                const float keep = up ? v[C / 2 + j] : v[j];
                v[j] = keep + __shfl_xor_sync(kFull, send, O);
            }
            if constexpr (O > 1) Butterfly<O / 2, C / 2>::run(v, lane);
        } else {
            v[0] = v[0] + __shfl_xor_sync(kFull, v[0], O);
            if constexpr (O > 1) Butterfly<O / 2, 1>::run(v, lane);
        }
    }
};

template <int Q>
__device__ __forceinline__ void reduce_scatter(float (&v)[Q], int lane)
{
    static_assert(Q >= 1 && Q <= 32 && (Q & (Q - 1)) == 0, "Q must be a power of two <= 32");
    Butterfly<16, Q>::run(v, lane);
}

// Programmatic dependent launch.  A kernel may read weights (never written by this
// library's kernels) before pdl_wait(); everything a preceding kernel may have
// produced or may still read (activations, routing, scales, outputs, workspace) is
// touched only after it.  pdl_wait() returns at once when the launch had no
// programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Pull `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Greedy-pick order: larger value first, then lower index; NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void set_status(uint8_t* ws, int bits)
{
    atomicOr(reinterpret_cast<int*>(ws + kWsStatus), bits);
}

}  // namespace dg
