// dg_tc_head.cu -- tcgen05 tensor-core family (DG_VAR_TC) for the fp8 vocabulary
// head with the fused greedy pick (mstar PR #1102, "What changed": an fp8 copy of
// the head with one scale for all of it; the pick at temperature 0 in the graph).
//
// From 2 token rows the CUDA-core head is bound by fp8 decode and FMA issue, so the
// contraction moves to the tensor cores with kind::f8f6f4 and the e4m3 weights go
// from HBM to the MMA untouched (TMA, 128-byte swizzle, no dequantisation).
// The bf16 activations are brought to e4m3 without losing their value:
//   sigma_t = 2^(7 - floor(log2 max_k |x[t,k]|))   (scaled magnitudes below 256)
//   y = x * sigma_t (exact), hi = e4m3(y), lo = e4m3(y - hi)
// A bf16 value has 8 significant bits and an e4m3 value 4, so y - hi (exact in
// fp32) is exactly representable as lo whenever |y| >= 1/4; below that e4m3's
// subnormal spacing 2^-9 limits lo, i.e. an absolute error of at most 2^-10 in the
// scaled domain (4.4e-6 * max|x| per element).  One MMA with N = 16 multiplies a
// 128-row weight tile with the 8 "hi" rows and the 8 "lo" rows of the tokens;
//   logit[t, n] = ((D[n, t] + D[n, 8 + t]) / sigma_t) * scale
// so this family's result is exact up to that floor and fp32 accumulation, and
// its variants (pipeline depth) share one arithmetic.
//   warp 0       TMA producer of 128x128 e4m3 weight boxes (ring of stages)
//   warp 1       TMEM allocation; lane 0 issues the MMAs into two accumulators
//   warps 1..5   build the split activations in shared memory (once per CTA)
//   warps 2..5   epilogue: TMEM -> logits (bf16) and per-token running pick
// Persistent CTAs (one per SM) walk the 128-row tiles; the CTA partial picks go
// through the workspace and the last CTA to arrive folds them (atomic ticket).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "dg_internal.h"
#include "dg_tc_common.cuh"

namespace dg {
namespace {

constexpr int kRows = 128;                 // weight rows per tile (MMA M)
constexpr int kKB = 128;                   // e4m3 elements (bytes) per stage row
constexpr int kWBox = kRows * kKB;         // 16 KB
constexpr int kTokens = 8;                 // token rows per launch
constexpr int kBRows = 2 * kTokens;        // hi + lo rows (MMA N)
constexpr int kXBlock = kBRows * kKB;      // 2 KB of split activations per k-block
constexpr int kThreads = 192;

struct HeadArgs {
    int N, K, M;
    int tiles, nkb, stages;
    const uint16_t* x;
    const float* scale;
    uint16_t* logits;       // may be null
    int32_t* argmax;
    uint8_t* ws;
};

// kind::f8f6f4 instruction descriptor: e4m3 A and B, fp32 accumulate, N = 16, M = 128.
constexpr uint32_t kIdesc = tc::idesc_f8(kBRows);

__global__ void __launch_bounds__(kThreads, 1)
    tc_head_kernel(const __grid_constant__ CUtensorMap tmW, HeadArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = a.stages;
    uint8_t* xsplit = smem;                                        // nkb blocks of 2 KB (SW128, 16 rows)
    uint8_t* wst = smem + static_cast<size_t>(a.nkb) * kXBlock;   // S stages of 16 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(wst + static_cast<size_t>(S) * kWBox);
    // bars: full[S], empty[S], accf[2], acce[2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    __shared__ float inv_sigma[kTokens];
    __shared__ float redmax[5][kTokens];
    __shared__ float sv[4][kTokens];
    __shared__ int si[4][kTokens];
    __shared__ int last_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = tc::su32(bars), empty0 = tc::su32(bars + S), accf0 = tc::su32(bars + 2 * S),
                   acce0 = tc::su32(bars + 2 * S + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::bar_init(full0 + 8 * s, 1);
            tc::bar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::bar_init(accf0 + 8 * b, 1);
            tc::bar_init(acce0 + 8 * b, 4);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(tc::su32(tmem_holder)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_holder;
    pdl_launch_dependents();

    // Tiles of this CTA: blockIdx.x, blockIdx.x + G, ...
    const int G = gridDim.x;
    const int my_tiles = a.tiles > static_cast<int>(blockIdx.x) ? (a.tiles - 1 - blockIdx.x) / G + 1 : 0;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t once = tc::policy_evict_first();   // weights are read exactly once
            int i = 0;
            bool stop = false;
            for (int jt = 0; jt < my_tiles && !stop; ++jt) {
                const int tile = blockIdx.x + jt * G;
                for (int kb = 0; kb < a.nkb; ++kb, ++i) {
                    const int s = i % S;
                    const uint32_t round = static_cast<uint32_t>(i / S);
                    if (!tc::bar_wait(empty0 + 8 * s, (round & 1u) ^ 1u, abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc::bar_expect_tx(full0 + 8 * s, kWBox);
                    tc::tma_2d_hint(tc::su32(wst + s * kWBox), &tmW, kb * kKB, tile * kRows, full0 + 8 * s, once);
                }
            }
        }
    } else {
        // ------------------------------------------------------- split activations
        pdl_wait();
        const int t160 = threadIdx.x - 32;                       // 0..159 over warps 1..5
        // 1) per-token max |x|
        for (int t = 0; t < kTokens; ++t) {
            float m = 0.0f;
            if (t < a.M)
                for (int v8 = t160; v8 < a.K / 8; v8 += 160) {
                    const uint4 q = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.K + v8 * 8);
                    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w4[j])), fabsf(bf16_hi(w4[j]))));
                }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
            if (lane == 0) redmax[warp - 1][t] = m;
        }
        asm volatile("bar.sync 1, 160;" ::: "memory");
        if (t160 < kTokens) {
            float m = 0.0f;
            for (int w = 0; w < 5; ++w) m = fmaxf(m, redmax[w][t160]);
            // sigma = 2^(7 - floor(log2 m)); the scaled maximum lies in [128, 256).
            const int e = tc::split_exponent(m);
            inv_sigma[t160] = ldexpf(1.0f, -e);
            redmax[0][t160] = ldexpf(1.0f, e);                   // sigma itself
        }
        asm volatile("bar.sync 1, 160;" ::: "memory");
        // 2) hi / lo e4m3 rows in the 128-byte-swizzled K-major layout:
        //    k-block kb, row r (0..7 hi, 8..15 lo), 16-byte chunk c at
        //    kb*2048 + (r/8)*1024 + (r%8)*128 + ((c ^ (r%8)) * 16).
        const int chunks = a.nkb * kTokens * 8;                  // (kb, token, chunk)
        for (int q = t160; q < chunks; q += 160) {
            const int c = q & 7, t = (q >> 3) % kTokens, kb = q / (8 * kTokens);
            uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
            if (t < a.M) tc::split_chunk(a.x + static_cast<size_t>(t) * a.K, kb * kKB + c * 16, a.K, redmax[0][t], hi, lo);
            uint8_t* blk = xsplit + kb * kXBlock;
            *reinterpret_cast<uint4*>(blk + tc::sw128_offset(t, c)) = hi;
            *reinterpret_cast<uint4*>(blk + tc::sw128_offset(kTokens + t, c)) = lo;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> MMA reads
        asm volatile("bar.sync 1, 160;" ::: "memory");

        if (warp == 1) {
            // -------------------------------------------------------------- MMA issue
            if (lane == 0) {
                int i = 0;
                bool stop = false;
                for (int jt = 0; jt < my_tiles && !stop; ++jt) {
                    const int b = jt & 1;
                    const uint32_t use = static_cast<uint32_t>(jt >> 1);
                    if (!tc::bar_wait(acce0 + 8 * b, (use & 1u) ^ 1u, abort_flag)) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + static_cast<uint32_t>(b * kBRows);
                    for (int kb = 0; kb < a.nkb; ++kb, ++i) {
                        const int s = i % S;
                        const uint32_t round = static_cast<uint32_t>(i / S);
                        if (!tc::bar_wait(full0 + 8 * s, round & 1u, abort_flag)) {
                            stop = true;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t wa = tc::su32(wst + s * kWBox), xa = tc::su32(xsplit + kb * kXBlock);
#pragma unroll
                        for (int kk = 0; kk < kKB / 32; ++kk)
                            tc::mma_f8(d, tc::sw128_desc(wa + kk * 32), tc::sw128_desc(xa + kk * 32), kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                        tc::commit(empty0 + 8 * s);
                    }
                    tc::commit(accf0 + 8 * b);
                }
            }
        } else {
            // -------------------------------------------------------------- epilogue
            const int q = warp & 3;
            const int row = q * 32 + lane;
            const float scale = *a.scale;
            float isg[kTokens];
#pragma unroll
            for (int t = 0; t < kTokens; ++t) isg[t] = inv_sigma[t];
            float best_v[kTokens];
            int best_i[kTokens];
#pragma unroll
            for (int t = 0; t < kTokens; ++t) {
                best_v[t] = -INFINITY;
                best_i[t] = 0x7fffffff;
            }
            for (int jt = 0; jt < my_tiles; ++jt) {
                const int b = jt & 1;
                const uint32_t use = static_cast<uint32_t>(jt >> 1);
                if (!tc::bar_wait(accf0 + 8 * b, use & 1u, abort_flag)) break;
                tc::fence_after();
                uint32_t v[16];
                tc::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kBRows), v);
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::bar_arrive(acce0 + 8 * b);
                const int n = (blockIdx.x + jt * G) * kRows + row;
                if (n < a.N) {
#pragma unroll
                    for (int t = 0; t < kTokens; ++t) {
                        if (t >= a.M) break;
                        const float dsum = __uint_as_float(v[t]) + __uint_as_float(v[kTokens + t]);
                        const float logit = (dsum * isg[t]) * scale;
                        if (a.logits) a.logits[static_cast<size_t>(t) * a.N + n] = f32_to_bf16_bits(logit);
                        if (better(logit, n, best_v[t], best_i[t])) {
                            best_v[t] = logit;
                            best_i[t] = n;
                        }
                    }
                }
            }
            // Per-token pick over this CTA, then across CTAs (last CTA by ticket).
#pragma unroll
            for (int t = 0; t < kTokens; ++t)
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const float ov = __shfl_xor_sync(kFull, best_v[t], o);
                    const int oi = __shfl_xor_sync(kFull, best_i[t], o);
                    if (better(ov, oi, best_v[t], best_i[t])) {
                        best_v[t] = ov;
                        best_i[t] = oi;
                    }
                }
            if (lane == 0)
#pragma unroll
                for (int t = 0; t < kTokens; ++t) {
                    sv[q][t] = best_v[t];
                    si[q][t] = best_i[t];
                }
            asm volatile("bar.sync 2, 128;" ::: "memory");
            float* pv = reinterpret_cast<float*>(a.ws + kWsData);
            int* pi = reinterpret_cast<int*>(a.ws + kWsData) + static_cast<size_t>(gridDim.x) * kTokens;
            const int et = threadIdx.x - 64;
            if (et < kTokens) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int w = 0; w < 4; ++w)
                    if (better(sv[w][et], si[w][et], bv, bi)) {
                        bv = sv[w][et];
                        bi = si[w][et];
                    }
                pv[blockIdx.x * kTokens + et] = bv;
                pi[blockIdx.x * kTokens + et] = bi;
            }
            __threadfence();
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (et == 0) last_sh = atomicAdd(reinterpret_cast<unsigned*>(a.ws + kWsTicket), 1u) == gridDim.x - 1;
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (last_sh) {
                __threadfence();
                // All 128 epilogue threads fold the CTA partials, one token at a time.
                for (int t = 0; t < a.M; ++t) {
                    float bv = -INFINITY;
                    int bi = 0x7fffffff;
                    for (int c = et; c < static_cast<int>(gridDim.x); c += 128) {
                        const float vv = ld_cg_f32(pv + c * kTokens + t);
                        const int ii = ld_cg_s32(pi + c * kTokens + t);
                        if (better(vv, ii, bv, bi)) {
                            bv = vv;
                            bi = ii;
                        }
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        const float ov = __shfl_xor_sync(kFull, bv, o);
                        const int oi = __shfl_xor_sync(kFull, bi, o);
                        if (better(ov, oi, bv, bi)) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    if (lane == 0) {
                        sv[q][0] = bv;
                        si[q][0] = bi;
                    }
                    asm volatile("bar.sync 2, 128;" ::: "memory");
                    if (et == 0) {
                        for (int w = 0; w < 4; ++w)
                            if (better(sv[w][0], si[w][0], bv, bi)) {
                                bv = sv[w][0];
                                bi = si[w][0];
                            }
                        a.argmax[t] = (bi == 0x7fffffff) ? -1 : bi;
                    }
                    asm volatile("bar.sync 2, 128;" ::: "memory");
                }
                if (et == 0) *reinterpret_cast<unsigned*>(a.ws + kWsTicket) = 0u;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

}  // namespace

// Shared memory of one CTA for K and `stages` (0 when it cannot fit).
size_t tc_head_smem(int K, int stages)
{
    const size_t nkb = (K + kKB - 1) / kKB;
    return 1024 + nkb * kXBlock + static_cast<size_t>(stages) * kWBox + (2 * stages + 4) * 8 + 16;
}

dg_status launch_tc_head(const DeviceInfo* dev, const dg_choice& c, const void* x, const void* Wq,
                         const float* scale, void* logits, int32_t* argmax, int M, int N, int K, void* ws,
                         size_t ws_bytes, cudaStream_t stream)
{
    if (M < 1 || M > kTokens) return DG_ERR_UNSUPPORTED_SHAPE;
    int stages = c.params[0];
    if (stages == 0) {
        stages = 2;
        while (stages < 16 && tc_head_smem(K, stages + 1) <= kMaxDynSmem) ++stages;
    }
    if (stages < 2 || stages > 16 || tc_head_smem(K, stages) > kMaxDynSmem) return DG_ERR_BAD_VARIANT;
    const int grid = dev->sm_count;
    if (ws_bytes < kWsData + static_cast<size_t>(grid) * kTokens * 8) return DG_ERR_WORKSPACE_TOO_SMALL;
    std::call_once(g_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    });
    if (!g_encode) return DG_ERR_CUDA;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {kKB, kRows};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Wq), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DG_ERR_CUDA;
    HeadArgs a{};
    a.N = N;
    a.K = K;
    a.M = M;
    a.tiles = (N + kRows - 1) / kRows;
    a.nkb = (K + kKB - 1) / kKB;
    a.stages = stages;
    a.x = static_cast<const uint16_t*>(x);
    a.scale = scale;
    a.logits = static_cast<uint16_t*>(logits);
    a.argmax = argmax;
    a.ws = static_cast<uint8_t*>(ws);
    const void* fn = reinterpret_cast<const void*>(&tc_head_kernel);
    const size_t smem = tc_head_smem(K, stages);
    if (occupancy(fn, kThreads, smem) < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    void* args[] = {&tm, &a};
    if (launch_kernel(fn, static_cast<unsigned>(grid), kThreads, smem, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg
