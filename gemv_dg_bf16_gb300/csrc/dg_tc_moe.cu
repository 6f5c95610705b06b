// dg_tc_moe.cu -- tcgen05 tensor-core family (DG_VAR_TC) of the routed-expert
// GEMMs: W1 + SiLU.mul and W2 + gate-weighted combine ("Decode optimization
// round 3", "Retained change 1: N-split W1/W2 MoE kernels").
//
// The experts' e4m3 rows stream from HBM through TMA (128-byte swizzle) straight
// into tcgen05.mma kind::f8f6f4; the (token, slot) pairs of an expert -- at most 8
// per pass -- enter as the exact hi/lo e4m3 split of their bf16 activation rows
// (power-of-two row scale; the same split as the fp8 head, error bounded by the
// e4m3 subnormal floor), so one N = 16 MMA serves 8 pairs x 2 pieces.
// Work units are (active expert, 128-row tile) in expert-major order; each
// persistent CTA takes one contiguous range of units, so it rebuilds the split
// activations only when its expert (or pair chunk) changes.
//   W1 tile: 64 gate rows j0.. and the 64 matching up rows I + j0.. (two TMA boxes);
//            a[t, k, j] = bf16(silu(g * s1[e, j]) * (u * s1[e, I + j]))
//   W2 tile: 128 output rows n0..; (h * s2[e, n]) * gw[t, k] go to the workspace;
//            after one grid barrier (one CTA per SM, launched cooperatively so all
//            are resident at once) every CTA folds a share of the outputs over the
//            valid slots in slot order.
//   warp 0     TMA producer (weights only, ring of stages)
//   warp 1     TMEM allocation, MMA issue (lane 0)
//   warps 2-5  split activations for each pass, epilogue of each tile
// Every mbarrier wait is bounded and flags DG_DEVERR_WAIT_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "dg_internal.h"
#include "dg_moe.cuh"
#include "dg_tc_common.cuh"

namespace dg {
namespace {

using namespace tc;

constexpr int kRows = 128;               // MMA M (weight rows per tile)
constexpr int kKB = 128;                 // e4m3 elements per stage row
constexpr int kWBox = kRows * kKB;       // 16 KB
constexpr int kPairs = 8;                // pairs per pass
constexpr int kBRows = 2 * kPairs;       // hi + lo rows (MMA N)
constexpr int kXBlock = kBRows * kKB;    // 2 KB of split activations per k-block
constexpr int kThreads = 192;
constexpr uint32_t kIdesc = idesc_f8(kBRows);

struct TcMoeArgs {
    MoeArgs m;
    int T;          // tiles per expert
    int nkb;        // k-blocks
    int stages;
};

template <bool W1>
__global__ void __launch_bounds__(kThreads, 1)
    tc_moe_kernel(const __grid_constant__ CUtensorMap tmW, TcMoeArgs A)
{
    const MoeArgs& a = A.m;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = A.stages;
    uint8_t* xsplit = smem;                                        // nkb x 2 KB
    uint8_t* wst = smem + static_cast<size_t>(A.nkb) * kXBlock;   // S x 16 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(wst + static_cast<size_t>(S) * kWBox);
    // full[S], empty[S], accf[2], acce[2], xready
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    __shared__ Route R;
    __shared__ float red[4][kPairs];
    __shared__ float sig[kPairs], isig[kPairs];
    __shared__ float exch[kPairs][64];       // W1: up values of a tile's 64 columns
    __shared__ int grid_ok;                   // W2: the grid barrier completed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();                               // routing and activations come from earlier kernels
    route_scan(R, a.ids, a.M, a.topk, a.E, a.ws);

    const uint32_t full0 = su32(bars), empty0 = su32(bars + S), accf0 = su32(bars + 2 * S),
                   acce0 = su32(bars + 2 * S + 2), xready = su32(bars + 2 * S + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            bar_init(full0 + 8 * s, 1);
            bar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(accf0 + 8 * b, 1);
            bar_init(acce0 + 8 * b, 4);
        }
        bar_init(xready, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(su32(tmem_holder)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_holder;

    // This CTA's contiguous range of (expert, tile) units.
    const int T = A.T;
    const long units = static_cast<long>(R.U) * T;
    const int u0 = static_cast<int>(blockIdx.x * units / gridDim.x);
    const int u1 = static_cast<int>((blockIdx.x + 1) * units / gridDim.x);
    const int rows_per_e = W1 ? 2 * a.I : a.Nout;
    const int kdim = a.K;                     // W1: hidden; W2: I

    // Passes: (expert, pair chunk) x the CTA's tiles of that expert.
    auto for_each_pass = [&](auto&& body) {
        for (int u = u0; u < u1;) {
            const int ue = u / T;
            const int t_lo = u - ue * T;
            const int t_hi = min(T, u1 - ue * T);
            for (int p0 = R.offs[ue]; p0 < R.offs[ue + 1]; p0 += kPairs)
                if (!body(ue, p0, min(kPairs, R.offs[ue + 1] - p0), t_lo, t_hi)) return;
            u = ue * T + t_hi;
        }
    };

    if (warp == 0) {
        // -------------------------------------------------------------------- producer
        if (lane == 0) {
            int i = 0;
            for_each_pass([&](int ue, int, int, int t_lo, int t_hi) {
                const int e = R.experts[ue];
                for (int tile = t_lo; tile < t_hi; ++tile)
                    for (int kb = 0; kb < A.nkb; ++kb, ++i) {
                        const int s = i % S;
                        const uint32_t round = static_cast<uint32_t>(i / S);
                        if (!bar_wait(empty0 + 8 * s, (round & 1u) ^ 1u, abort_flag)) return false;
                        bar_expect_tx(full0 + 8 * s, kWBox);
                        const uint32_t dst = su32(wst + s * kWBox);
                        if constexpr (W1) {
                            tma_2d(dst, &tmW, kb * kKB, e * rows_per_e + tile * 64, full0 + 8 * s);
                            tma_2d(dst + kWBox / 2, &tmW, kb * kKB, e * rows_per_e + a.I + tile * 64, full0 + 8 * s);
                        } else {
                            tma_2d(dst, &tmW, kb * kKB, e * rows_per_e + tile * kRows, full0 + 8 * s);
                        }
                    }
                return true;
            });
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA
        if (lane == 0) {
            int i = 0, jt = 0, pass = 0;
            for_each_pass([&](int, int, int, int t_lo, int t_hi) {
                if (!bar_wait(xready, static_cast<uint32_t>(pass & 1), abort_flag)) return false;
                ++pass;
                fence_after();
                for (int tile = t_lo; tile < t_hi; ++tile, ++jt) {
                    const int b = jt & 1;
                    const uint32_t use = static_cast<uint32_t>(jt >> 1);
                    if (!bar_wait(acce0 + 8 * b, (use & 1u) ^ 1u, abort_flag)) return false;
                    fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(b * kBRows);
                    for (int kb = 0; kb < A.nkb; ++kb, ++i) {
                        const int s = i % S;
                        const uint32_t round = static_cast<uint32_t>(i / S);
                        if (!bar_wait(full0 + 8 * s, round & 1u, abort_flag)) return false;
                        fence_after();
                        const uint32_t wa = su32(wst + s * kWBox), xa = su32(xsplit + kb * kXBlock);
#pragma unroll
                        for (int kk = 0; kk < kKB / 32; ++kk)
                            mma_f8(d, sw128_desc(wa + kk * 32), sw128_desc(xa + kk * 32), kIdesc,
                                   (kb > 0 || kk > 0) ? 1u : 0u);
                        commit(empty0 + 8 * s);
                    }
                    commit(accf0 + 8 * b);
                }
                return true;
            });
        }
    } else {
        // ------------------------------------------------- split activations + epilogue
        const int et = threadIdx.x - 64;          // 0..127
        const int q = warp & 3;                   // TMEM lane quarter
        const int row = q * 32 + lane;
        float* terms = reinterpret_cast<float*>(a.ws + kWsData);
        int jt = 0;
        for_each_pass([&](int ue, int p0, int c, int t_lo, int t_hi) {
            const int e = R.experts[ue];
            // (1) row maxima of the chunk's activation rows
            for (int p = 0; p < kPairs; ++p) {
                float m = 0.0f;
                if (p < c) {
                    const int t = R.ptok[p0 + p], k = R.pslot[p0 + p];
                    const uint16_t* src = a.x + (W1 ? static_cast<size_t>(t) : static_cast<size_t>(t) * a.topk + k) *
                                                    static_cast<size_t>(kdim);
                    for (int v8 = et; v8 < kdim / 8; v8 += 128) {
                        const uint4 qv = *reinterpret_cast<const uint4*>(src + v8 * 8);
                        const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w4[j])), fabsf(bf16_hi(w4[j]))));
                    }
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
                if (lane == 0) red[q][p] = m;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et < kPairs) {
                const float m = fmaxf(fmaxf(red[0][et], red[1][et]), fmaxf(red[2][et], red[3][et]));
                const int ex = split_exponent(m);
                sig[et] = ldexpf(1.0f, ex);
                isig[et] = ldexpf(1.0f, -ex);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            // (2) hi / lo rows into the swizzled layout (rows p and 8 + p of each k-block)
            const int chunks = A.nkb * kPairs * 8;
            for (int qq = et; qq < chunks; qq += 128) {
                const int ch = qq & 7, p = (qq >> 3) % kPairs, kb = qq / (8 * kPairs);
                uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (p < c) {
                    const int t = R.ptok[p0 + p], k = R.pslot[p0 + p];
                    const uint16_t* src = a.x + (W1 ? static_cast<size_t>(t) : static_cast<size_t>(t) * a.topk + k) *
                                                    static_cast<size_t>(kdim);
                    split_chunk(src, kb * kKB + ch * 16, kdim, sig[p], hi, lo);
                }
                uint8_t* blk = xsplit + kb * kXBlock;
                *reinterpret_cast<uint4*>(blk + sw128_offset(p, ch)) = hi;
                *reinterpret_cast<uint4*>(blk + sw128_offset(kPairs + p, ch)) = lo;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et == 0) bar_arrive(xready);
            float is[kPairs];
#pragma unroll
            for (int p = 0; p < kPairs; ++p) is[p] = isig[p];

            // (3) epilogue of each tile of the pass
            for (int tile = t_lo; tile < t_hi; ++tile, ++jt) {
                const int b = jt & 1;
                const uint32_t use = static_cast<uint32_t>(jt >> 1);
                if (!bar_wait(accf0 + 8 * b, use & 1u, abort_flag)) return false;
                fence_after();
                uint32_t v[16];
                tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kBRows), v);
                fence_before();
                __syncwarp();
                if (lane == 0) bar_arrive(acce0 + 8 * b);
                if constexpr (W1) {
                    const int jl = row & 63;
                    const int j = tile * 64 + jl;
                    const bool up = row >= 64;
                    const float sc = j < a.I ? a.s[static_cast<size_t>(e) * 2 * a.I + (up ? a.I : 0) + j] : 0.0f;
                    if (up)
#pragma unroll
                        for (int p = 0; p < kPairs; ++p)
                            exch[p][jl] = ((__uint_as_float(v[p]) + __uint_as_float(v[kPairs + p])) * is[p]) * sc;
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (!up && j < a.I)
                        for (int p = 0; p < c; ++p) {
                            const float g = ((__uint_as_float(v[p]) + __uint_as_float(v[kPairs + p])) * is[p]) * sc;
                            const float silu = g / (1.0f + expf(-g));
                            const int t = R.ptok[p0 + p], k = R.pslot[p0 + p];
                            a.out[(static_cast<size_t>(t) * a.topk + k) * a.I + j] = f32_to_bf16_bits(silu * exch[p][jl]);
                        }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                } else {
                    const int n = tile * kRows + row;
                    if (n < a.Nout) {
                        const float s2 = a.s[static_cast<size_t>(e) * a.Nout + n];
                        for (int p = 0; p < c; ++p) {
                            const int t = R.ptok[p0 + p], k = R.pslot[p0 + p];
                            const float h = ((__uint_as_float(v[p]) + __uint_as_float(v[kPairs + p])) * is[p]) * s2;
                            terms[(static_cast<size_t>(t) * a.topk + k) * a.Nout + n] = h * a.gw[t * a.topk + k];
                        }
                    }
                }
            }
            return true;
        });
        if constexpr (W1) {
            // Invalid slots get a = 0 (no unit covers them), written by CTA 0.
            if (blockIdx.x == 0)
                for (int i = 0; i < a.M * a.topk; ++i)
                    if (!R.valid[i])
                        for (int j = et; j < a.I; j += 128) a.out[static_cast<size_t>(i) * a.I + j] = 0;
        } else {
            // Combine: once every CTA has written its terms (one grid barrier; the grid
            // is one CTA per SM and the launch is cooperative, so all are resident), the
            // outputs are folded in slot order, spread over every CTA's epilogue
            // threads.  Tokens without a valid slot get y = 0.
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et == 0) grid_ok = grid_barrier(reinterpret_cast<unsigned*>(a.ws + kWsGridBarrier), abort_flag) ? 1 : 0;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (grid_ok) {
                __threadfence();
                const long total = static_cast<long>(a.M) * a.Nout;
                for (long i = static_cast<long>(blockIdx.x) * 128 + et; i < total; i += static_cast<long>(gridDim.x) * 128) {
                    const int t = static_cast<int>(i / a.Nout), n = static_cast<int>(i - static_cast<long>(t) * a.Nout);
                    float y = 0.0f;
                    bool first = true;
                    for (int k = 0; k < a.topk; ++k) {
                        if (!R.valid[t * a.topk + k]) continue;
                        const float tv = ld_cg_f32(terms + (static_cast<size_t>(t) * a.topk + k) * a.Nout + n);
                        y = first ? tv : y + tv;
                        first = false;
                    }
                    a.out[static_cast<size_t>(t) * a.Nout + n] = f32_to_bf16_bits(y);
                }
            } else {
                // The barrier gave up: this CTA's share of y becomes NaN rather than
                // keeping an earlier call's values, beside the status word.
                const long total = static_cast<long>(a.M) * a.Nout;
                for (long i = static_cast<long>(blockIdx.x) * 128 + et; i < total; i += static_cast<long>(gridDim.x) * 128)
                    a.out[i] = 0x7FC0u;
                if (et == 0) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

size_t smem_bytes(int nkb, int stages)
{
    return 1024 + static_cast<size_t>(nkb) * kXBlock + static_cast<size_t>(stages) * kWBox + (2 * stages + 5) * 8 + 16;
}

}  // namespace

dg_status launch_tc_moe(bool w1, const DeviceInfo* dev, const dg_choice& c, const MoeArgs& m, cudaStream_t stream)
{
    const int kdim = m.K;
    const int nkb = (kdim + kKB - 1) / kKB;
    int stages = c.params[0];
    if (stages == 0) {
        stages = 2;
        while (stages < 16 && smem_bytes(nkb, stages + 1) <= kMaxDynSmem) ++stages;
    }
    if (stages < 2 || stages > 16 || smem_bytes(nkb, stages) > kMaxDynSmem) return DG_ERR_BAD_VARIANT;
    if (w1 && m.I % 64 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    const int T = w1 ? m.I / 64 : (m.Nout + kRows - 1) / kRows;
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
    const uint64_t rows = static_cast<uint64_t>(m.E) * (w1 ? 2 * m.I : m.Nout);
    CUtensorMap tm;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim)};
    const cuuint32_t box[2] = {kKB, static_cast<cuuint32_t>(w1 ? 64 : kRows)};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(m.W), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DG_ERR_CUDA;
    TcMoeArgs A{};
    A.m = m;
    A.T = T;
    A.nkb = nkb;
    A.stages = stages;
    const void* fn = w1 ? reinterpret_cast<const void*>(&tc_moe_kernel<true>)
                        : reinterpret_cast<const void*>(&tc_moe_kernel<false>);
    const size_t smem = smem_bytes(nkb, stages);
    if (occupancy(fn, kThreads, smem) < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    void* args[] = {&tm, &A};
    // W2 combines after a grid-wide barrier: launched cooperatively, so all its CTAs are
    // resident at once even when other streams' kernels hold SMs.
    const cudaError_t le = w1 ? launch_kernel(fn, static_cast<unsigned>(dev->sm_count), kThreads, smem, stream, args)
                              : launch_kernel_cooperative(fn, static_cast<unsigned>(dev->sm_count), kThreads, smem,
                                                          stream, args);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg
