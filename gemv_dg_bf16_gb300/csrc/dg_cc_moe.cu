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
#include "dg_tc_common.cuh"

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

// ------------------------------------------------------------------ row ranges
// The same outputs in the same arithmetic, cut the other way: CTA b owns one
// contiguous range of rows of EVERY active expert, so no output is shared between
// CTAs.  W2: output rows n in [lo, hi); each (slot, n) term stays in shared memory and
// the CTA folds y[t, n] over the valid slots in slot order at the end -- no ticket,
// no fence, no pass through the workspace.  W1 has no combine: the CTA takes a
// contiguous share of the flattened (active expert, column pair) list, so the share
// is even to one column pair whatever the expert count.  The activation rows (W2:
// all M x topk rows of a; W1: the M rows of x) do not depend on the routing: one bulk
// copy brings them into shared memory while the routing is built.  A warp loads two K segments of its rows before folding the first, which
// halves the dependent memory round trips of an item.

// Canonical-order partial of segment s for R rows x MT pairs whose activation rows sit
// anywhere in shared memory (xr[t] = pair t's row): fold_segment's arithmetic with the
// activation rows gathered instead of strided.
template <int MT, int R>
__device__ __forceinline__ void fold_gathered(const uint4 (&w)[kSeg / (32 * WTraits<WT_E4M3>::VE)][R], int K, int s,
                                              const uint4* const (&xr)[MT], int lane, float& total)
{
    constexpr int VE = WTraits<WT_E4M3>::VE;
    constexpr int VPS = kSeg / (32 * VE);
    constexpr int MTP = cpow2(MT);
    constexpr int Q = R * MTP;
    float p[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) p[q] = 0.0f;
#pragma unroll
    for (int v = 0; v < VPS; ++v) {
        const int k = s * kSeg + v * (32 * VE) + lane * VE;
        if (k >= K) continue;
        // 16 e4m3 weights = two halves of 8, each against one bf16 vector of x
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 xv[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) xv[t] = xr[t][k / 8 + h];
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
                        const uint32_t wword = (&w[v][r].x)[2 * h + ww];
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
    reduce_scatter<Q>(p, lane);
    total = (s == 0) ? p[0] : total + p[0];
}

// Row total over all segments: for one pair two segments' loads in flight at a time,
// for more pairs one (the accumulators need the registers).
template <int MT, int R>
__device__ __forceinline__ float gathered_total(const uint8_t* const (&wrow)[R], const bool (&rok)[R], int K,
                                                const uint4* const (&xr)[MT], int lane)
{
    constexpr int VPS = kSeg / (32 * WTraits<WT_E4M3>::VE);
    const int nseg = (K + kSeg - 1) / kSeg;
    float total = 0.0f;
    if constexpr (MT > 1) {
        for (int s = 0; s < nseg; ++s) {
            uint4 w0[VPS][R];
            load_segment<WT_E4M3, R>(w0, wrow, rok, K, s, lane);
            fold_gathered<MT, R>(w0, K, s, xr, lane, total);
        }
    } else {
        for (int s = 0; s < nseg; s += 2) {
            uint4 w0[VPS][R], w1[VPS][R];
            load_segment<WT_E4M3, R>(w0, wrow, rok, K, s, lane);
            if (s + 1 < nseg) load_segment<WT_E4M3, R>(w1, wrow, rok, K, s + 1, lane);
            fold_gathered<MT, R>(w0, K, s, xr, lane, total);
            if (s + 1 < nseg) fold_gathered<MT, R>(w1, K, s + 1, xr, lane, total);
        }
    }
    return total;
}

// Shared-memory layout of the row-range kernel, the same on host and device:
// activation rows (W2: the M x topk rows of a; W1: the M rows of x), then W2's terms
// [M x topk slots][rows per CTA].
__host__ __device__ inline size_t range_xs_bytes(bool w1, int M, int topk, int K)
{
    return static_cast<size_t>(w1 ? M : M * topk) * K * 2;
}

__host__ __device__ inline size_t range_smem_bytes(bool w1, int M, int topk, int K, int rpc)
{
    return range_xs_bytes(w1, M, topk, K) + (w1 ? 0 : static_cast<size_t>(M) * topk * rpc * 4);
}

// One item: R rows of expert u for pairs [p0, p0 + MT), the emitted outputs as in
// w1_chunk / w2_chunk (W2's terms into shared memory instead of the workspace).
template <bool W1, int MT>
__device__ void range_item(const MoeArgs& a, const Route& R, int e, int r0, int p0, const uint4* xs,
                           float* terms, int lo, int hi, int rpc)
{
    constexpr int RH = kMoeR / 2;
    constexpr int MTP = cpow2(MT);
    constexpr int Q = kMoeR * MTP;
    constexpr int SH = 5 - clog2(Q);
    const int lane = threadIdx.x & 31;
    const int idx = lane >> SH, my_r = idx / MTP, my_t = idx % MTP;
    const int kv = a.K / 8;
    const uint4* xr[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t)
        xr[t] = xs + static_cast<size_t>(W1 ? R.ptok[p0 + t] : R.ptok[p0 + t] * a.topk + R.pslot[p0 + t]) * kv;
    const uint8_t* wrow[kMoeR];
    bool rok[kMoeR];
    if constexpr (W1) {
        // r0 = first column j of the item; rows j, j+1 (gate) and I+j, I+j+1 (up)
        const uint8_t* We = a.W + static_cast<size_t>(e) * 2 * a.I * a.K;
#pragma unroll
        for (int r = 0; r < kMoeR; ++r) {
            const int j = r0 + (r % RH);
            rok[r] = j < a.I;
            wrow[r] = We + static_cast<size_t>((r < RH ? 0 : a.I) + (rok[r] ? j : r0)) * a.K;
        }
        const float total = gathered_total<MT, kMoeR>(wrow, rok, a.K, xr, lane);
        const float up = __shfl_sync(kFull, total, (lane + ((RH * MTP) << SH)) & 31);
        const int j = r0 + my_r;
        const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT && my_r < RH;
        if (writer && j < a.I) {
            const float g = total * a.s[static_cast<size_t>(e) * 2 * a.I + j];
            const float u = up * a.s[static_cast<size_t>(e) * 2 * a.I + a.I + j];
            const float silu = g / (1.0f + expf(-g));
            const int t = R.ptok[p0 + my_t], k = R.pslot[p0 + my_t];
            a.out[(static_cast<size_t>(t) * a.topk + k) * a.I + j] = f32_to_bf16_bits(silu * u);
        }
    } else {
        // r0 = first output row n of the item (rows n < hi of this CTA's range)
        const uint8_t* We = a.W + static_cast<size_t>(e) * a.Nout * a.K;
#pragma unroll
        for (int r = 0; r < kMoeR; ++r) {
            rok[r] = r0 + r < hi;
            wrow[r] = We + static_cast<size_t>(rok[r] ? r0 + r : lo) * a.K;
        }
        const float total = gathered_total<MT, kMoeR>(wrow, rok, a.K, xr, lane);
        const int n = r0 + my_r;
        const bool writer = (lane & ((1 << SH) - 1)) == 0 && my_t < MT;
        if (writer && n < hi) {
            const int t = R.ptok[p0 + my_t], k = R.pslot[p0 + my_t];
            const float h = total * a.s[static_cast<size_t>(e) * a.Nout + n];
            terms[(t * a.topk + k) * rpc + (n - lo)] = h * a.gw[t * a.topk + k];
        }
    }
}

template <bool W1, int MTMAX>
__device__ void range_items(int c, const MoeArgs& a, const Route& R, int e, int r0, int p0, const uint4* xs,
                            float* terms, int lo, int hi, int rpc)
{
#define DG_MOE_CASE(MT)                                                                    \
    case MT:                                                                               \
        if constexpr (MT <= MTMAX) range_item<W1, MT>(a, R, e, r0, p0, xs, terms, lo, hi, rpc); \
        break;
    switch (c) {
        DG_MOE_CASE(1) DG_MOE_CASE(2) DG_MOE_CASE(3) DG_MOE_CASE(4)
        DG_MOE_CASE(5) DG_MOE_CASE(6) DG_MOE_CASE(7) DG_MOE_CASE(8)
    default: break;
    }
#undef DG_MOE_CASE
}

template <bool W1, int MTMAX>
__global__ void __launch_bounds__(256, 2) moe_range_kernel(MoeArgs a)
{
    __shared__ Route R;
    __shared__ __align__(8) uint64_t xbar;        // the activation copy's completion
    __shared__ int abort_s;
    extern __shared__ __align__(128) uint4 xs[];
    pdl_launch_dependents();
    pdl_wait();                                    // routing and activations come from earlier kernels
    const int kv = a.K / 8;
    const int P_all = a.M * a.topk;
    // The slot ids first (their latency overlaps the rest of the prologue), then one
    // bulk copy of every activation row the call can use, in row order (W2: the
    // M x topk rows of a, row t * topk + k; W1: the M rows of x), then the routing.
    const int e_lane = P_all <= 32 ? route_warp_load(a.ids, P_all) : -1;
    if (threadIdx.x == 0) {
        abort_s = 0;
        const uint32_t bar = tc::su32(&xbar);
        tc::bar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bytes = static_cast<uint32_t>(range_xs_bytes(W1, a.M, a.topk, a.K));
        tc::bar_expect_tx(bar, bytes);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         tc::su32(xs)),
                     "l"(a.x), "r"(bytes), "r"(bar)
                     : "memory");
    }
    if (P_all <= 32) route_warp_build(R, e_lane, a.M, a.topk, a.E, a.ws);
    else route_scan(R, a.ids, a.M, a.topk, a.E, a.ws);

    const int warp = threadIdx.x >> 5, wpc = blockDim.x >> 5;
    constexpr int RH = kMoeR / 2;
    // This CTA's share.  W2: rows [lo, hi) of every expert (rpc = a.tile rows per CTA,
    // the grid = ceil(Nout / rpc)).  W1: items [it_lo, it_hi) of the list (active
    // expert u, column pair jg), u-major.
    const int rpc = W1 ? 0 : a.tile;
    const int lo = W1 ? 0 : blockIdx.x * rpc;
    const int hi = W1 ? 0 : min(a.Nout, lo + rpc);
    const int ipe = W1 ? (a.I + RH - 1) / RH : (rpc + kMoeR - 1) / kMoeR;      // items per expert
    int it_lo, it_hi;                              // at most 1024 experts x 4096 items
    if constexpr (W1) {
        const long long n = static_cast<long long>(R.U) * ipe;
        it_lo = static_cast<int>(n * blockIdx.x / gridDim.x);
        it_hi = static_cast<int>(n * (blockIdx.x + 1) / gridDim.x);
    } else {
        it_lo = 0;
        it_hi = lo < hi ? R.U * ipe : 0;
    }
    if constexpr (W1) {
        // invalid slots get a = 0: this CTA clears its share of the columns
        const int j_lo = static_cast<int>(static_cast<long long>(a.I) * blockIdx.x / gridDim.x);
        const int j_hi = static_cast<int>(static_cast<long long>(a.I) * (blockIdx.x + 1) / gridDim.x);
        for (int i = 0; i < a.M * a.topk; ++i)
            if (!R.valid[i])
                for (int j = j_lo + threadIdx.x; j < j_hi; j += blockDim.x) a.out[static_cast<size_t>(i) * a.I + j] = 0;
    }
    if (threadIdx.x == 0) tc::bar_wait(tc::su32(&xbar), 0, &abort_s);
    __syncthreads();
    if (abort_s) {                                 // the activation copy never landed
        if (threadIdx.x == 0) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
        return;
    }
    float* terms = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + range_xs_bytes(W1, a.M, a.topk, a.K));

    for (int it = it_lo + warp; it < it_hi; it += wpc) {
        const int u = it / ipe, g = it - u * ipe;
        const int e = R.experts[u];
        const int r0 = W1 ? g * RH : lo + g * kMoeR;
        if (!W1 && r0 >= hi) continue;                 // the last CTA's short range
        const int pb = R.offs[u], pe = R.offs[u + 1];
        for (int p0 = pb; p0 < pe; p0 += MTMAX)
            range_items<W1, MTMAX>(min(MTMAX, pe - p0), a, R, e, r0, p0, xs, terms, lo, hi, rpc);
    }
    if constexpr (!W1) {
        __syncthreads();
        // y[t, n] = the valid slots' terms folded in slot order (0 for a token with none)
        const int w = hi - lo;
        for (int i = threadIdx.x; i < a.M * w; i += blockDim.x) {
            const int t = i / w, n = lo + (i - t * w);
            float y = 0.0f;
            bool first = true;
            for (int k = 0; k < a.topk; ++k) {
                if (!R.valid[t * a.topk + k]) continue;
                const float v = terms[(t * a.topk + k) * rpc + (n - lo)];
                y = first ? v : y + v;
                first = false;
            }
            a.out[static_cast<size_t>(t) * a.Nout + n] = f32_to_bf16_bits(y);
        }
    }
}

}  // namespace

size_t moe_range_smem(bool w1, int M, int topk, int K, int rpc) { return range_smem_bytes(w1, M, topk, K, rpc); }

const void* moe_range_kernel_fn(bool w1, int mtmax)
{
    switch (mtmax) {
    case 1: return w1 ? reinterpret_cast<const void*>(&moe_range_kernel<true, 1>)
                      : reinterpret_cast<const void*>(&moe_range_kernel<false, 1>);
    case 2: return w1 ? reinterpret_cast<const void*>(&moe_range_kernel<true, 2>)
                      : reinterpret_cast<const void*>(&moe_range_kernel<false, 2>);
    case 4: return w1 ? reinterpret_cast<const void*>(&moe_range_kernel<true, 4>)
                      : reinterpret_cast<const void*>(&moe_range_kernel<false, 4>);
    case 8: return w1 ? reinterpret_cast<const void*>(&moe_range_kernel<true, 8>)
                      : reinterpret_cast<const void*>(&moe_range_kernel<false, 8>);
    default: return nullptr;
    }
}

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
