// dg_a8.cuh -- activation quantisation of the A8W8 block-scaled linear, shared by the
// tensor-core kernel's prologue and the standalone quantisation entry point.
//
// "Decode optimization round 3", "Retained change 2" (A8W8 blockscale GEMM rows at
// decode M) and "Rejected paths" / "Remaining headroom" (the quantisation kernels
// fused into the GEMM as a prologue).  Per token and 128-wide K-block, in binary32:
//   amax = max(max |x|, 2^-32),  r = 448 / amax,  sx = amax / 448,
//   q    = e4m3(x * r), round to nearest even, saturating at 448.
// Eight consecutive lanes hold one block, 16 elements (one 16-byte code chunk) each.
#pragma once

#include "dg_tc_common.cuh"

namespace dg {

constexpr int kA8Block = 128;              // K elements per scale block (and per 128 x 128 weight block)
constexpr float kA8Floor = 0x1p-32f;       // smallest block maximum (all-zero blocks give zero codes)

// 16 bf16 values (two 16-byte pieces, element order) as fp32.
__device__ __forceinline__ void a8_unpack16(const uint4& a, const uint4& b, float (&v)[16])
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
}

// Elements k0 .. k0+15 of a bf16 row as fp32; zeros from K on (K % 16 == 0).
__device__ __forceinline__ void a8_load16(const uint16_t* row, int k0, int K, float (&v)[16])
{
    if (k0 < K) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + k0);
        const uint4 b = *reinterpret_cast<const uint4*>(row + k0 + 8);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16_lo(w[i]);
            v[2 * i + 1] = bf16_hi(w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
}

// Block maximum: the chunk maxima of the 8 lanes sharing a block (lane bits 0..2),
// raised to the floor.  Every lane of the warp must call it.
__device__ __forceinline__ float a8_block_amax(const float (&v)[16])
{
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    return fmaxf(m, kA8Floor);
}

// The 16 codes e4m3(v[i] * r), element i in byte i.
__device__ __forceinline__ uint4 a8_codes(const float (&v)[16], float r)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = tc::to_e4m3x2(__fmul_rn(v[4 * i], r), __fmul_rn(v[4 * i + 1], r));
        const uint32_t hi = tc::to_e4m3x2(__fmul_rn(v[4 * i + 2], r), __fmul_rn(v[4 * i + 3], r));
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float a8_recip_scale(float amax) { return __fdiv_rn(448.0f, amax); }
__device__ __forceinline__ float a8_scale(float amax) { return __fdiv_rn(amax, 448.0f); }

}  // namespace dg
