// dg_cc_moe.cu -- small-M routed-expert GEMMs (W1 + SiLU.mul, W2 + combine) on
// CUDA cores, split along N.
//
// "Decode optimization round 3", "Retained change 1: N-split W1/W2 MoE kernels":
// at one to a few tokens only ~6 experts are active, so one CTA per expert (a
// full-N tile) leaves most of the GPU idle; the experts' rows are instead cut
// into many narrow N-tiles.  Here a work unit is (active expert, N-tile) and
// persistent CTAs walk the unit list.  Routing is recomputed by every CTA from
// topk_ids in shared memory (no host sync, no extra launch):
//   a slot (t, k) is valid when 0 <= id < E and no earlier slot of t names id;
//   active experts are listed in ascending id order; each expert's (token, slot)
//   pairs are listed by ascending token then slot.
// Arithmetic per output follows the canonical order of dg_common.cuh (e4m3
// weights, 16 per vector).  W2's per-slot terms go through the workspace and
// the CTA that finishes the last slot of a (token, N-tile) folds them in slot
// order, so the combine is deterministic and needs no waiting.
#include "dg_cc_dense.cuh"
#include "dg_internal.h"
#include "dg_moe.cuh"

namespace dg {

namespace {

constexpr int kMoeR = 4;             // rows per warp group
// Stage `c` activation rows (one per pair, `kv` 16-byte vectors each) into xs.
__device__ __forceinline__ void stage_rows(uint4* xs, const uint16_t* __restrict__ src,
                                           const Route& R, int p0, int c, int kv, bool w1, int topk,
                                           int K)
{
    for (int i = threadIdx.x; i < c * kv; i += blockDim.x) {
        const int q = i / kv, v = i - q * kv;
        const int t = R.ptok[p0 + q], k = R.pslot[p0 + q];
        const size_t row = w1 ? static_cast<size_t>(t) : static_cast<size_t>(t) * topk + k;
        xs[i] = *reinterpret_cast<const uint4*>(src + row * K + v * 8);
    }
}

// W1 unit body for a chunk of MT pairs: gate rows j and up rows I + j of expert e.
template <int MT>
__device__ void w1_chunk(const MoeArgs& a, const Route& R, int e, int j_lo, int j_hi, int p0,
                         const uint4* xs)
{
    constexpr int RH = kMoeR / 2;         // gate rows per group (and up rows)
    constexpr int MTP = cpow2(MT);
    constexpr int Q = kMoeR * MTP;
    constexpr int SH = 5 - clog2(Q);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpc = blockDim.x >> 5;
    const int idx = lane >> SH, my_r = idx / MTP, my_t = idx % MTP;
    const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT && my_r < RH;
    const int kv = a.K / 8;
    const uint8_t* We = a.W + static_cast<size_t>(e) * 2 * a.I * a.K;
    for (int j0 = j_lo + warp * RH; j0 < j_hi; j0 += wpc * RH) {
        const uint8_t* wrow[kMoeR];
        bool rok[kMoeR];
#pragma unroll
        for (int r = 0; r < kMoeR; ++r) {
            const int j = j0 + (r % RH);
            rok[r] = j < j_hi;
            const int row = (r < RH ? 0 : a.I) + (rok[r] ? j : j_lo);
            wrow[r] = We + static_cast<size_t>(row) * a.K;
        }
        const float total = row_group_total<WT_E4M3, MT, kMoeR>(wrow, rok, a.K, xs, kv, lane);
        // up partner of gate output (r, t) is (r + RH, t)
        const float up = __shfl_sync(kFull, total, (lane + ((RH * MTP) << SH)) & 31);
        const int j = j0 + my_r;
        if (writer && j < j_hi) {
            const float g = total * a.s[static_cast<size_t>(e) * 2 * a.I + j];
            const float u = up * a.s[static_cast<size_t>(e) * 2 * a.I + a.I + j];
            const float silu = g / (1.0f + expf(-g));
            const int t = R.ptok[p0 + my_t], k = R.pslot[p0 + my_t];
            a.out[(static_cast<size_t>(t) * a.topk + k) * a.I + j] = f32_to_bf16_bits(silu * u);
        }
    }
}

// W2 unit body for a chunk of MT pairs: rows n of expert e, terms to workspace.
template <int MT>
__device__ void w2_chunk(const MoeArgs& a, const Route& R, int e, int n_lo, int n_hi, int p0,
                         const uint4* xs, float* terms)
{
    constexpr int MTP = cpow2(MT);
    constexpr int Q = kMoeR * MTP;
    constexpr int SH = 5 - clog2(Q);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpc = blockDim.x >> 5;
    const int idx = lane >> SH, my_r = idx / MTP, my_t = idx % MTP;
    const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT;
    const int kv = a.K / 8;   // K here is I (the W2 reduction length)
    const uint8_t* We = a.W + static_cast<size_t>(e) * a.Nout * a.K;
    for (int n0 = n_lo + warp * kMoeR; n0 < n_hi; n0 += wpc * kMoeR) {
        const uint8_t* wrow[kMoeR];
        bool rok[kMoeR];
#pragma unroll
        for (int r = 0; r < kMoeR; ++r) {
            rok[r] = n0 + r < n_hi;
            wrow[r] = We + static_cast<size_t>(rok[r] ? n0 + r : n_lo) * a.K;
        }
        const float total = row_group_total<WT_E4M3, MT, kMoeR>(wrow, rok, a.K, xs, kv, lane);
        const int n = n0 + my_r;
        if (writer && n < n_hi) {
            const int t = R.ptok[p0 + my_t], k = R.pslot[p0 + my_t];
            const float h = total * a.s[static_cast<size_t>(e) * a.Nout + n];
            const float term = h * a.gw[t * a.topk + k];
            terms[(static_cast<size_t>(t) * a.topk + k) * a.Nout + n] = term;
        }
    }
}

template <bool W1, int MTMAX>
__device__ void run_chunk(int c, const MoeArgs& a, const Route& R, int e, int lo, int hi, int p0,
                          const uint4* xs, float* terms)
{
#define DG_MOE_CASE(MT)                                                       \
    case MT:                                                                  \
        if constexpr (MT <= MTMAX) {                                          \
            if constexpr (W1) w1_chunk<MT>(a, R, e, lo, hi, p0, xs);          \
            else w2_chunk<MT>(a, R, e, lo, hi, p0, xs, terms);                \
        }                                                                     \
        break;
    switch (c) {
        DG_MOE_CASE(1) DG_MOE_CASE(2) DG_MOE_CASE(3) DG_MOE_CASE(4)
        DG_MOE_CASE(5) DG_MOE_CASE(6) DG_MOE_CASE(7) DG_MOE_CASE(8)
    default: break;
    }
#undef DG_MOE_CASE
}

// MTMAX: most (token, slot) pairs of one expert handled in one pass over its rows.
// An expert with more pairs is walked in several passes (its rows come from L2 again);
// a small MTMAX keeps registers, and so resident warps, in check.
template <bool W1, int MTMAX>
__global__ void __launch_bounds__(256, MTMAX <= 2 ? 3 : 2) moe_kernel(MoeArgs a)
{
    __shared__ Route R;
    __shared__ int8_t fold_tok[16];      // W2: pairs of the unit whose token this unit folds
    extern __shared__ uint4 xs[];        // [MTMAX][K/8]
    pdl_launch_dependents();
    pdl_wait();                          // routing and activations come from earlier kernels
    route_scan(R, a.ids, a.M, a.topk, a.E, a.ws);

    const int rows = W1 ? a.I : a.Nout;                 // N-tiles cut these rows (W1: columns j)
    const int tiles = (rows + a.tile - 1) / a.tile;
    const int units = R.U * tiles;
    const int kv = a.K / 8;
    float* terms = reinterpret_cast<float*>(a.ws + kWsData);
    unsigned* tickets = reinterpret_cast<unsigned*>(a.ws + kWsCounters);

    if constexpr (W1) {
        // Invalid slots get a = 0 (no unit covers them).
        if (blockIdx.x == 0)
            for (int i = 0; i < a.M * a.topk; ++i)
                if (!R.valid[i])
                    for (int j = threadIdx.x; j < a.I; j += blockDim.x) a.out[static_cast<size_t>(i) * a.I + j] = 0;
    } else {
        // Tokens without a valid slot get y = 0 (nothing else writes them).
        if (blockIdx.x == 0)
            for (int t = 0; t < a.M; ++t)
                if (R.nvalid[t] == 0)
                    for (int n = threadIdx.x; n < a.Nout; n += blockDim.x) a.out[static_cast<size_t>(t) * a.Nout + n] = 0;
    }

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int ue = u / tiles, tile = u - ue * tiles;
        const int e = R.experts[ue];
        const int lo = tile * a.tile, hi = min(rows, lo + a.tile);
        const int pb = R.offs[ue], pe = R.offs[ue + 1];
        for (int p0 = pb; p0 < pe; p0 += MTMAX) {
            const int c = min(MTMAX, pe - p0);
            __syncthreads();                               // xs reuse
            stage_rows(xs, a.x, R, p0, c, kv, W1, a.topk, a.K);
            __syncthreads();
            run_chunk<W1, MTMAX>(c, a, R, e, lo, hi, p0, xs, terms);
        }
        if constexpr (!W1) {
            // Publish this unit's terms, then take every pair's (token, N-tile) ticket at
            // once (one thread per pair; an expert's pairs are distinct tokens); the
            // tokens whose last term this was are folded in slot order.
            __threadfence();
            __syncthreads();
            for (int p = pb + threadIdx.x; p < pe; p += blockDim.x) {
                const int t = R.ptok[p];
                const unsigned old = atomicAdd(&tickets[t * tiles + tile], 1u);
                fold_tok[p - pb] = (old + 1 == static_cast<unsigned>(R.nvalid[t])) ? 1 : 0;
            }
            __syncthreads();
            bool any = false;
            for (int p = pb; p < pe; ++p) {
                if (!fold_tok[p - pb]) continue;
                if (!any) __threadfence();
                any = true;
                const int t = R.ptok[p];
                for (int n = lo + threadIdx.x; n < hi; n += blockDim.x) {
                    float y = 0.0f;
                    bool first = true;
                    for (int k = 0; k < a.topk; ++k) {
                        if (!R.valid[t * a.topk + k]) continue;
                        const float v = ld_cg_f32(terms + (static_cast<size_t>(t) * a.topk + k) * a.Nout + n);
                        y = first ? v : y + v;
                        first = false;
                    }
                    a.out[static_cast<size_t>(t) * a.Nout + n] = f32_to_bf16_bits(y);
                }
                if (threadIdx.x == 0) tickets[t * tiles + tile] = 0u;
            }
            __syncthreads();                               // fold_tok reuse
        }
    }
}

}  // namespace

const void* moe_w1_kernel(int mtmax)
{
    switch (mtmax) {
    case 1: return reinterpret_cast<const void*>(&moe_kernel<true, 1>);
    case 2: return reinterpret_cast<const void*>(&moe_kernel<true, 2>);
    case 4: return reinterpret_cast<const void*>(&moe_kernel<true, 4>);
    case 8: return reinterpret_cast<const void*>(&moe_kernel<true, 8>);
    default: return nullptr;
    }
}

const void* moe_w2_kernel(int mtmax)
{
    switch (mtmax) {
    case 1: return reinterpret_cast<const void*>(&moe_kernel<false, 1>);
    case 2: return reinterpret_cast<const void*>(&moe_kernel<false, 2>);
    case 4: return reinterpret_cast<const void*>(&moe_kernel<false, 4>);
    case 8: return reinterpret_cast<const void*>(&moe_kernel<false, 8>);
    default: return nullptr;
    }
}

}  // namespace dg
