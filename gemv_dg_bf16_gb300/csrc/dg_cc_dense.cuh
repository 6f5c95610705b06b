// dg_cc_dense.cuh -- CUDA-core family (DG_VAR_CC_WARP) for the dense ops:
// bf16 linear, fused gate/up + SiLU.mul, fp8 head + greedy argmax.
//
// Geometry: each warp owns groups of R consecutive weight rows; a group is
// streamed once through registers with 16-byte non-allocating loads (all
// R x VPS vectors of a segment are in flight together) while the activations
// of MT tokens sit in shared memory as bf16.  CTAs are persistent: warps walk
// the row groups with a grid-wide stride.  The arithmetic is the canonical
// order described in dg_common.cuh, so R, warps per CTA and grid size change
// only speed, never bits.
#pragma once

#include "dg_common.cuh"

namespace dg {

enum : int { EPI_STORE = 0, EPI_GATEUP = 1, EPI_HEAD = 2 };
enum : int { WT_BF16 = 0, WT_E4M3 = 1 };

struct DenseArgs {
    const uint8_t* W;       // [N, K] weights (bf16 bits or e4m3 codes)
    const uint16_t* x;      // [M_total, K] bf16 activations
    int N;                  // weight rows
    int K;
    int t0;                 // first token of this launch's chunk
    int groups;             // ceil(N / R)
    int ksplit;             // KSPLIT kernels: warps sharing one row group's segments (2, 4 or 8; divides wpc)
    uint16_t* out;          // bf16 output: y [M, N], gate/up out [M, N/2], or head logits (may be null)
    int ld_out;             // output row stride in elements
    const float* scale;     // head: per-tensor scale (device)
    int32_t* argmax;        // head: [M]
    uint8_t* ws;            // workspace
};

template <int WT>
struct WTraits;
template <>
struct WTraits<WT_BF16> {
    static constexpr int VE = 8;      // weights per 16-byte vector
    static constexpr int ESZ = 2;
};
template <>
struct WTraits<WT_E4M3> {
    static constexpr int VE = 16;
    static constexpr int ESZ = 1;
};

// Accumulate one 16-byte weight vector of each of R rows into p for MT tokens.
// xs points at this lane's x vectors (token stride xstride uint4s); elements are
// consumed in ascending order j = 0..VE-1, as CO requires.
template <int WT, int MT, int R, int MTP>
__device__ __forceinline__ void fma_vector(const uint4 (&w)[R], const uint4* xs, int xstride,
                                           float (&p)[R * MTP])
{
    if constexpr (WT == WT_BF16) {
        // bf16 x bf16 products are exact in fp32, so the mixed-precision fma (bf16
        // operands, fp32 addend, one rounding) gives the same bits as converting
        // both operands to fp32 first -- without the conversions.
        uint4 xv[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) xv[t] = xs[t * xstride];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t ww = (&w[r].x)[wd];
#pragma unroll
                for (int t = 0; t < MT; ++t) fma2_bf16(p[r * MTP + t], (&xv[t].x)[wd], ww);
            }
        }
    } else {
        // 16 e4m3 weights = two 8-element halves, each matching one x vector.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 xv[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) xv[t] = xs[t * xstride + h];
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    float x0[MT], x1[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const uint32_t xw = (&xv[t].x)[2 * ww + pp];
                        x0[t] = bf16_lo(xw);
                        x1[t] = bf16_hi(xw);
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t wword = (&w[r].x)[2 * h + ww];
                        const float2 wf = e4m3x2_to_f32(pp ? (wword >> 16) : wword);
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
                            float acc = p[r * MTP + t];
                            acc = __fmaf_rn(x0[t], wf.x, acc);
                            acc = __fmaf_rn(x1[t], wf.y, acc);
                            p[r * MTP + t] = acc;
                        }
                    }
                }
            }
        }
    }
}

// Load this lane's VPS vectors of segment s for R rows (zero outside the matrix).
template <int WT, int R>
__device__ __forceinline__ void load_segment(uint4 (&w)[kSeg / (32 * WTraits<WT>::VE)][R],
                                             const uint8_t* const (&wrow)[R], const bool (&rok)[R], int K,
                                             int s, int lane)
{
    using T = WTraits<WT>;
    constexpr int VE = T::VE;
    constexpr int VPS = kSeg / (32 * VE);
#pragma unroll
    for (int v = 0; v < VPS; ++v) {
        const int k = s * kSeg + v * (32 * VE) + lane * VE;
#pragma unroll
        for (int r = 0; r < R; ++r)
            w[v][r] = (rok[r] && k < K) ? ld_stream(wrow[r] + static_cast<size_t>(k) * T::ESZ)
                                        : make_uint4(0, 0, 0, 0);
    }
}

// Canonical-order partial of segment s (lane chains, then the butterfly): lanes
// with idx = lane >> SH return the partial of output idx.
template <int WT, int MT, int R>
__device__ __forceinline__ float segment_partial(const uint4 (&w)[kSeg / (32 * WTraits<WT>::VE)][R], int K, int s,
                                                 const uint4* xs_smem, int xstride, int lane)
{
    constexpr int VE = WTraits<WT>::VE;
    constexpr int VPS = kSeg / (32 * VE);
    constexpr int MTP = cpow2(MT);
    constexpr int Q = R * MTP;
    float p[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) p[q] = 0.0f;
#pragma unroll
    for (int v = 0; v < VPS; ++v) {
        const int k = s * kSeg + v * (32 * VE) + lane * VE;
        if (k < K) fma_vector<WT, MT, R, MTP>(w[v], xs_smem + k / 8, xstride, p);
    }
    reduce_scatter<Q>(p, lane);
    return p[0];
}

// Canonical-order partial of segment s (lane chains, then the butterfly), folded
// into `total`.
template <int WT, int MT, int R>
__device__ __forceinline__ void fold_segment(const uint4 (&w)[kSeg / (32 * WTraits<WT>::VE)][R], int K, int s,
                                             const uint4* xs_smem, int xstride, int lane, float& total)
{
    constexpr int VE = WTraits<WT>::VE;
    constexpr int VPS = kSeg / (32 * VE);
    constexpr int MTP = cpow2(MT);
    constexpr int Q = R * MTP;
    float p[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) p[q] = 0.0f;
#pragma unroll
    for (int v = 0; v < VPS; ++v) {
        const int k = s * kSeg + v * (32 * VE) + lane * VE;
        if (k < K) fma_vector<WT, MT, R, MTP>(w[v], xs_smem + k / 8, xstride, p);
    }
    reduce_scatter<Q>(p, lane);
    total = (s == 0) ? p[0] : total + p[0];
}

// One row group: returns this lane's folded total for output index
// idx = lane >> SH, i.e. (r = idx / MTP, t = idx % MTP).  (Loading segment s + 1
// before reducing segment s was measured on GB300: it costs occupancy and loses
// more than it hides, most of all for e4m3 rows.)
template <int WT, int MT, int R>
__device__ __forceinline__ float row_group_total(const uint8_t* const (&wrow)[R],
                                                 const bool (&rok)[R], int K,
                                                 const uint4* xs_smem, int xstride, int lane)
{
    constexpr int VPS = kSeg / (32 * WTraits<WT>::VE);
    const int nseg = (K + kSeg - 1) / kSeg;
    float total = 0.0f;
    for (int s = 0; s < nseg; ++s) {
        uint4 w[VPS][R];
        load_segment<WT, R>(w, wrow, rok, K, s, lane);
        fold_segment<WT, MT, R>(w, K, s, xs_smem, xstride, lane, total);
    }
    return total;
}

template <int WT, int MT, int R, int EPI, bool KSPLIT>
__global__ void __launch_bounds__(256) cc_dense_kernel(DenseArgs a)
{
    constexpr int MTP = cpow2(MT);
    constexpr int Q = R * MTP;
    constexpr int SH = 5 - clog2(Q);
    static_assert(Q <= 32, "rows x tokens per warp must fit one warp reduction");
    static_assert(EPI != EPI_GATEUP || (R % 2) == 0, "gate/up needs row pairs");

    extern __shared__ uint4 xs[];               // [MT][K/8] bf16 vectors
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wpc = blockDim.x >> 5;
    const int kv = a.K / 8;

    // Weights only: start the first segment of this warp's first row group on its way
    // into L2 while a preceding kernel may still be finishing, then wait for it.
    {
        const int g0 = blockIdx.x * wpc + warp;
        const int row = g0 * R + lane;
        if (lane < R && g0 < a.groups && row < a.N)
            prefetch_l2(a.W + static_cast<size_t>(row) * a.K * WTraits<WT>::ESZ,
                        static_cast<uint32_t>(min(a.K, kSeg) * WTraits<WT>::ESZ));
    }
    pdl_launch_dependents();
    pdl_wait();

    // Stage this chunk's activations.
    for (int i = threadIdx.x; i < MT * kv; i += blockDim.x) {
        const int t = i / kv, c = i - t * kv;
        xs[i] = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(a.t0 + t) * a.K + c * 8);
    }
    __syncthreads();

    const int idx = lane >> SH;
    const int my_r = idx / MTP;
    const int my_t = idx % MTP;
    const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT;

    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    float scale = 1.0f;
    if constexpr (EPI == EPI_HEAD) scale = *a.scale;

    // Per row group: `total` -> the op's output (and the head's running pick).
    auto emit = [&](int row0, float total) {
        const int row = row0 + my_r;
        if constexpr (EPI == EPI_STORE) {
            if (writer && row < a.N)
                a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row] = f32_to_bf16_bits(total);
        } else if constexpr (EPI == EPI_GATEUP) {
            // The up row of pair (2j, 2j+1) sits MTP outputs further on.
            const float u = __shfl_sync(kFull, total, (lane + (MTP << SH)) & 31);
            if (writer && (my_r % 2) == 0 && row < a.N) {
                const float g_ = total;
                const float silu = g_ / (1.0f + expf(-g_));
                a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row / 2] =
                    f32_to_bf16_bits(silu * u);
            }
        } else {
            const float logit = total * scale;
            if (writer && row < a.N) {
                if (a.out)
                    a.out[static_cast<size_t>(a.t0 + my_t) * a.ld_out + row] = f32_to_bf16_bits(logit);
                if (better(logit, row, best_v, best_i)) {
                    best_v = logit;
                    best_i = row;
                }
            }
        }
    };

    if constexpr (!KSPLIT) {
        for (int g = blockIdx.x * wpc + warp; g < a.groups; g += gridDim.x * wpc) {
            const int row0 = g * R;
            const uint8_t* wrow[R];
            bool rok[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                rok[r] = (row0 + r) < a.N;
                wrow[r] = a.W + static_cast<size_t>(rok[r] ? row0 + r : 0) * a.K * WTraits<WT>::ESZ;
            }
            emit(row0, row_group_total<WT, MT, R>(wrow, rok, a.K, xs, kv, lane));
        }
    } else {
        // K-split inside the CTA: the ksplit warps of a slot share one row group,
        // warp `part` taking segments part, part + ksplit, ...; the segment partials
        // meet in shared memory and are folded left in segment order by the slot's
        // first warp -- the same sums in the same order as one warp doing them all.
        constexpr int VPS = kSeg / (32 * WTraits<WT>::VE);
        const int ks = a.ksplit, slots = wpc / ks;
        const int slot = warp / ks, part = warp - slot * ks;
        const int nseg = (a.K + kSeg - 1) / kSeg;
        float* P = reinterpret_cast<float*>(xs + MT * kv) + static_cast<size_t>(slot) * nseg * Q;
        const int idx_w = lane >> SH;
        const bool idx_writer = (lane & ((1 << SH) - 1)) == 0;
        const int per_round = gridDim.x * slots;
        const int rounds = (a.groups + per_round - 1) / per_round;
        for (int rd = 0; rd < rounds; ++rd) {
            const int g = rd * per_round + blockIdx.x * slots + slot;
            const int row0 = g * R;
            if (g < a.groups) {
                const uint8_t* wrow[R];
                bool rok[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    rok[r] = (row0 + r) < a.N;
                    wrow[r] = a.W + static_cast<size_t>(rok[r] ? row0 + r : 0) * a.K * WTraits<WT>::ESZ;
                }
                for (int s = part; s < nseg; s += ks) {
                    uint4 w[VPS][R];
                    load_segment<WT, R>(w, wrow, rok, a.K, s, lane);
                    const float ps = segment_partial<WT, MT, R>(w, a.K, s, xs, kv, lane);
                    if (idx_writer) P[s * Q + idx_w] = ps;
                }
            }
            __syncthreads();
            if (part == 0 && g < a.groups) {
                float total = P[idx_w];
                for (int s = 1; s < nseg; ++s) total = total + P[s * Q + idx_w];
                emit(row0, total);
            }
            __syncthreads();
        }
    }

    if constexpr (EPI == EPI_HEAD) {
        // Warp: combine lanes that hold the same token (they differ in the r and
        // duplicate bits of the lane id, not in the token bits).
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
        __shared__ float sv[8][MTP];
        __shared__ int si[8][MTP];
        __shared__ bool last;
        if (my_r == 0 && (lane & ((1 << SH) - 1)) == 0) {
            sv[warp][my_t] = best_v;
            si[warp][my_t] = best_i;
        }
        __syncthreads();
        float* pv = reinterpret_cast<float*>(a.ws + kWsData);
        int* pi = reinterpret_cast<int*>(a.ws + kWsData) + static_cast<size_t>(gridDim.x) * MTP;
        if (threadIdx.x < MT) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int w2 = 0; w2 < wpc; ++w2)
                if (better(sv[w2][threadIdx.x], si[w2][threadIdx.x], bv, bi)) {
                    bv = sv[w2][threadIdx.x];
                    bi = si[w2][threadIdx.x];
                }
            pv[blockIdx.x * MTP + threadIdx.x] = bv;
            pi[blockIdx.x * MTP + threadIdx.x] = bi;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned* ticket = reinterpret_cast<unsigned*>(a.ws + kWsTicket);
            last = atomicAdd(ticket, 1u) == gridDim.x - 1;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
        // Last CTA: fold all CTA partials (the pick order is a total order, so
        // the result does not depend on which CTA arrived last).
        for (int t = 0; t < MT; ++t) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int c = threadIdx.x; c < gridDim.x; c += blockDim.x) {
                const float v = ld_cg_f32(pv + c * MTP + t);
                const int i = ld_cg_s32(pi + c * MTP + t);
                if (better(v, i, bv, bi)) {
                    bv = v;
                    bi = i;
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
            __syncthreads();
            if (threadIdx.x == 0) {
                for (int w2 = 1; w2 < wpc; ++w2)
                    if (better(sv[w2][0], si[w2][0], bv, bi)) {
                        bv = sv[w2][0];
                        bi = si[w2][0];
                    }
                a.argmax[a.t0 + t] = (bi == 0x7fffffff) ? -1 : bi;
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) *reinterpret_cast<unsigned*>(a.ws + kWsTicket) = 0u;
    }
}

}  // namespace dg
