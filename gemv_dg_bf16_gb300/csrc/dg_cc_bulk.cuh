// dg_cc_bulk.cuh -- CUDA-core family, bulk-copy staged variant (DG_VAR_CC_BULK).
//
// One persistent CTA per SM (or two).  CTA c owns the contiguous rows
// [c*N/G, (c+1)*N/G) (row pairs for gate/up), walked in blocks of 8*RW rows.  A
// producer warp streams each block's weight rows segment by segment into a ring
// of shared-memory stages with cp.async.bulk (1-D TMA; one copy per row segment,
// completion counted in bytes on the stage's mbarrier); eight consumer warps each
// own RW rows of the block and run exactly the canonical order of dg_common.cuh
// on the staged vectors (same per-lane chains, same butterfly, same left fold over
// segments), so this variant is bitwise identical to the register-streamed one.
// Deep staging keeps ~100-200 KB of weights in flight per SM without spending
// registers on it.  Every mbarrier wait is bounded (flag + wind down).
#pragma once

#include "dg_cc_dense.cuh"

namespace dg {

constexpr int kBulkConsumers = 8;
constexpr int kBulkThreads = (kBulkConsumers + 1) * 32;
constexpr unsigned long long kBulkWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t bulk_smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool bulk_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool bulk_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag)
{
    if (bulk_try(bar, parity)) return true;
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t i = 1;; ++i) {
        if (bulk_try(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (t - t0 > kBulkWaitNs) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <int WT, int MT, int RW, int EPI>
__global__ void __launch_bounds__(kBulkThreads, 1) cc_bulk_kernel(DenseArgs a, int stages)
{
    using T = WTraits<WT>;
    constexpr int VE = T::VE;
    constexpr int VPS = kSeg / (32 * VE);
    constexpr int SEGB = kSeg * T::ESZ;                  // bytes of one full row segment
    constexpr int RB = kBulkConsumers * RW;              // rows per block
    constexpr int STAGE = RB * SEGB;
    constexpr int MTP = cpow2(MT);
    constexpr int Q = RW * MTP;
    constexpr int SH = 5 - clog2(Q);
    static_assert(Q <= 32, "rows x tokens per warp must fit one warp reduction");
    static_assert(EPI != EPI_GATEUP || RW == 2, "gate/up warps own one (gate, up) row pair");

    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ int abort_sh;
    __shared__ float sv[kBulkConsumers][MTP];
    __shared__ int si[kBulkConsumers][MTP];
    __shared__ int last_sh;
    volatile int* abort_flag = &abort_sh;

    const int kv = a.K / 8;
    const size_t xbytes = (static_cast<size_t>(MT) * a.K * 2 + 127) / 128 * 128;
    uint4* xs = reinterpret_cast<uint4*>(smem_raw);
    uint8_t* stg = smem_raw + xbytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg + static_cast<size_t>(stages) * STAGE);
    const uint32_t full0 = bulk_smem_u32(bars), empty0 = bulk_smem_u32(bars + stages);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const long units = (EPI == EPI_GATEUP) ? a.N / 2 : a.N;
    const int upr = (EPI == EPI_GATEUP) ? 2 : 1;
    const int r_lo = static_cast<int>(blockIdx.x * units / G) * upr;
    const int r_hi = static_cast<int>((blockIdx.x + 1) * units / G) * upr;
    const int nblk = (r_hi - r_lo + RB - 1) / RB;
    const int nseg = (a.K + kSeg - 1) / kSeg;
    const int items = nblk * nseg;

    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * s), "r"(1));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty0 + 8 * s), "r"(kBulkConsumers));
        }
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    for (int i = threadIdx.x; i < MT * kv; i += blockDim.x) {
        const int t = i / kv, c = i - t * kv;
        xs[i] = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(a.t0 + t) * a.K + c * 8);
    }
    __syncthreads();

    if (warp == kBulkConsumers) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            for (int i = 0; i < items; ++i) {
                const int s = i % stages;
                const uint32_t round = static_cast<uint32_t>(i / stages);
                if (!bulk_wait(empty0 + 8 * s, (round & 1u) ^ 1u, abort_flag)) break;
                const int blk = i / nseg, seg = i - blk * nseg;
                const int row0 = r_lo + blk * RB;
                const int nr = min(RB, r_hi - row0);
                const int k0 = seg * kSeg;
                const uint32_t segbytes = static_cast<uint32_t>(min(kSeg, a.K - k0) * T::ESZ);
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full0 + 8 * s),
                             "r"(segbytes * nr)
                             : "memory");
                const uint32_t dst0 = bulk_smem_u32(stg + static_cast<size_t>(s) * STAGE);
                for (int r = 0; r < nr; ++r) {
                    const uint8_t* src = a.W + (static_cast<size_t>(row0 + r) * a.K + k0) * T::ESZ;
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            dst0 + r * SEGB),
                        "l"(src), "r"(segbytes), "r"(full0 + 8 * s)
                        : "memory");
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- consumers
        const int idx = lane >> SH, my_r = idx / MTP, my_t = idx % MTP;
        const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT;
        float scale = 1.0f;
        if constexpr (EPI == EPI_HEAD) scale = *a.scale;
        float best_v = -INFINITY;
        int best_i = 0x7fffffff;
        float total = 0.0f;
        for (int i = 0; i < items; ++i) {
            const int s = i % stages;
            const uint32_t round = static_cast<uint32_t>(i / stages);
            if (!bulk_wait(full0 + 8 * s, round & 1u, abort_flag)) break;
            const int blk = i / nseg, seg = i - blk * nseg;
            const int row0 = r_lo + blk * RB;
            const int nr = min(RB, r_hi - row0);
            const uint8_t* st = stg + static_cast<size_t>(s) * STAGE;
            bool rok[RW];
#pragma unroll
            for (int j = 0; j < RW; ++j) rok[j] = warp * RW + j < nr;
            float p[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) p[q] = 0.0f;
#pragma unroll
            for (int v = 0; v < VPS; ++v) {
                const int kk = v * (32 * VE) + lane * VE;          // offset inside the segment
                const int k = seg * kSeg + kk;
                if (k < a.K) {
                    uint4 w[RW];
#pragma unroll
                    for (int j = 0; j < RW; ++j)
                        w[j] = rok[j] ? *reinterpret_cast<const uint4*>(st + (warp * RW + j) * SEGB + kk * T::ESZ)
                                      : make_uint4(0, 0, 0, 0);
                    fma_vector<WT, MT, RW, MTP>(w, xs + k / 8, kv, p);
                }
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * s) : "memory");
            reduce_scatter<Q>(p, lane);
            total = (seg == 0) ? p[0] : total + p[0];
            if (seg == nseg - 1) {
                const int row = row0 + warp * RW + my_r;
                const bool ok_row = warp * RW + my_r < nr;
                if constexpr (EPI == EPI_STORE) {
                    if (writer && ok_row)
                        a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row] = f32_to_bf16_bits(total);
                } else if constexpr (EPI == EPI_GATEUP) {
                    const float u = __shfl_sync(kFull, total, (lane + (MTP << SH)) & 31);
                    if (writer && my_r == 0 && ok_row) {
                        const float silu = total / (1.0f + expf(-total));
                        a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row / 2] = f32_to_bf16_bits(silu * u);
                    }
                } else {
                    const float logit = total * scale;
                    if (writer && ok_row) {
                        if (a.out)
                            a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row] = f32_to_bf16_bits(logit);
                        if (better(logit, row, best_v, best_i)) {
                            best_v = logit;
                            best_i = row;
                        }
                    }
                }
            }
        }
        if constexpr (EPI == EPI_HEAD) {
            // Same pick reduction as the register-streamed variant, over the consumer warps.
            constexpr int TB_LO = SH, TB_HI = SH + clog2(MTP);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                if (o >= (1 << TB_LO) && o < (1 << TB_HI)) continue;
                const float ov = __shfl_xor_sync(kFull, best_v, o);
                const int oi = __shfl_xor_sync(kFull, best_i, o);
                if (better(ov, oi, best_v, best_i)) {
                    best_v = ov;
                    best_i = oi;
                }
            }
            if (my_r == 0 && (lane & ((1 << SH) - 1)) == 0) {
                sv[warp][my_t] = best_v;
                si[warp][my_t] = best_i;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kBulkConsumers * 32) : "memory");
            float* pv = reinterpret_cast<float*>(a.ws + kWsData);
            int* pi = reinterpret_cast<int*>(a.ws + kWsData) + static_cast<size_t>(gridDim.x) * MTP;
            if (threadIdx.x < MT) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int w2 = 0; w2 < kBulkConsumers; ++w2)
                    if (better(sv[w2][threadIdx.x], si[w2][threadIdx.x], bv, bi)) {
                        bv = sv[w2][threadIdx.x];
                        bi = si[w2][threadIdx.x];
                    }
                pv[blockIdx.x * MTP + threadIdx.x] = bv;
                pi[blockIdx.x * MTP + threadIdx.x] = bi;
            }
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"r"(kBulkConsumers * 32) : "memory");
            if (threadIdx.x == 0) {
                unsigned* ticket = reinterpret_cast<unsigned*>(a.ws + kWsTicket);
                last_sh = atomicAdd(ticket, 1u) == gridDim.x - 1;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kBulkConsumers * 32) : "memory");
            if (last_sh) {
                __threadfence();
                for (int t = 0; t < MT; ++t) {
                    float bv = -INFINITY;
                    int bi = 0x7fffffff;
                    for (int c = threadIdx.x; c < static_cast<int>(gridDim.x); c += kBulkConsumers * 32) {
                        const float v = ld_cg_f32(pv + c * MTP + t);
                        const int i2 = ld_cg_s32(pi + c * MTP + t);
                        if (better(v, i2, bv, bi)) {
                            bv = v;
                            bi = i2;
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
                        sv[warp][0] = bv;
                        si[warp][0] = bi;
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kBulkConsumers * 32) : "memory");
                    if (threadIdx.x == 0) {
                        for (int w2 = 1; w2 < kBulkConsumers; ++w2)
                            if (better(sv[w2][0], si[w2][0], bv, bi)) {
                                bv = sv[w2][0];
                                bi = si[w2][0];
                            }
                        a.argmax[a.t0 + t] = (bi == 0x7fffffff) ? -1 : bi;
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kBulkConsumers * 32) : "memory");
                }
                if (threadIdx.x == 0) *reinterpret_cast<unsigned*>(a.ws + kWsTicket) = 0u;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && abort_sh) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
}

}  // namespace dg
