// dg_moe.cuh -- argument block and workspace layout of the MoE kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "dg_common.cuh"

namespace dg {

struct MoeArgs {
    const uint16_t* x;      // W1: x [M, K]; W2: a [M, topk, I] (K = I)
    const int32_t* ids;     // [M, topk]
    const float* gw;        // W2: gate weights [M, topk]
    const uint8_t* W;       // W1 [E, 2I, K] or W2 [E, Nout, I] e4m3 codes
    const float* s;         // W1 [E, 2I] or W2 [E, Nout] row scales
    uint16_t* out;          // W1: a [M, topk, I]; W2: y [M, Nout]
    uint8_t* ws;
    int M, topk, E, I, K, Nout;
    int tile;               // N-tile: W1 columns j per unit, W2 rows n per unit
};

__host__ __device__ inline size_t moe_terms_bytes(int M, int topk, int Nout)
{
    return (static_cast<size_t>(M) * topk * Nout * 4 + 255) / 256 * 256;
}

__host__ __device__ inline int moe_tickets(int M, int Nout, int tile)
{
    return M * ((Nout + tile - 1) / tile);
}

// ---------------------------------------------------------------------- routing
// A slot (t, k) is valid when 0 <= id < E and no earlier slot of t names id;
// active experts are listed in ascending id order; each expert's (token, slot)
// pairs by ascending token then slot.  Every CTA derives the same tables.
constexpr int kMoeMaxPairs = 128;    // M * topk
constexpr int kMoeMaxE = 1024;

struct Route {
    int U;                           // active experts
    int P;                           // valid pairs
    int nvalid[16];                  // valid slots per token
    int16_t experts[kMoeMaxPairs];   // active expert ids, ascending
    int16_t offs[kMoeMaxPairs + 1];  // pairs of active expert u: [offs[u], offs[u+1])
    int8_t ptok[kMoeMaxPairs];
    int8_t pslot[kMoeMaxPairs];
    int8_t valid[kMoeMaxPairs];
    int cnt[kMoeMaxE];               // per expert: pair count, then pair offset
};

// Up to 32 slots: warp 0 builds every table, one slot per lane (one global load, no
// shared-memory passes over the experts, one barrier).  Lane i holds slot i = (t, k);
// its pair position is the number of valid slots with a smaller expert id plus the
// earlier valid slots of the same expert (ascending expert, then token, then slot);
// its expert's index is the number of distinct smaller experts.  The load and the
// build are separate steps so that a kernel can issue other copies in between.
__device__ __forceinline__ int route_warp_load(const int32_t* __restrict__ ids, int P_all)
{
    return (threadIdx.x < 32 && static_cast<int>(threadIdx.x) < P_all) ? ids[threadIdx.x] : -1;
}

__device__ inline void route_warp_build(Route& R, int e, int M, int topk, int E, uint8_t* ws)
{
    __shared__ int se[32];
    const int P_all = M * topk;
    if (threadIdx.x < 32) {
        const int i = threadIdx.x;
        const bool in = i < P_all;
        se[i] = e;
        __syncwarp();
        const int t = in ? i / topk : 0, k = in ? i - t * topk : 0;
        bool ok = in && e >= 0 && e < E;
        for (int j = 0; j < k; ++j)
            if (se[t * topk + j] == e) ok = false;
        const unsigned vmask = __ballot_sync(kFull, ok);
        int smaller = 0, same_before = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const int ej = se[j];
            const bool vj = (vmask >> j) & 1u;
            smaller += (vj && ej < e) ? 1 : 0;
            same_before += (vj && ej == e && j < i) ? 1 : 0;
        }
        const bool first = ok && same_before == 0;
        const unsigned fmask = __ballot_sync(kFull, first);
        int u = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) u += (((fmask >> j) & 1u) && se[j] < e) ? 1 : 0;
        if (in) R.valid[i] = ok ? 1 : 0;
        if (in && !ok && blockIdx.x == 0) set_status(ws, DG_DEVERR_BAD_TOPK_ID);
        if (ok) {
            const int pos = smaller + same_before;
            R.ptok[pos] = static_cast<int8_t>(t);
            R.pslot[pos] = static_cast<int8_t>(k);
            if (first) {
                R.experts[u] = static_cast<int16_t>(e);
                R.offs[u] = static_cast<int16_t>(smaller);
            }
        }
        const int U = __popc(fmask), P = __popc(vmask);
        if (i == 0) {
            R.U = U;
            R.P = P;
            R.offs[U] = static_cast<int16_t>(P);
        }
        if (i < M) {
            const unsigned tok = ((1u << topk) - 1u) << (i * topk);
            R.nvalid[i] = __popc(vmask & tok);
        }
    }
    __syncthreads();
}

// Every CTA computes the same routing tables (deterministic, no atomics on order).
// topk_ids is read from global memory once, into shared memory.
__device__ inline void route_scan(Route& R, const int32_t* __restrict__ ids, int M, int topk, int E,
                           uint8_t* ws)
{
    if (M * topk <= 32) {
        route_warp_build(R, route_warp_load(ids, M * topk), M, topk, E, ws);
        return;
    }
    __shared__ int sid[kMoeMaxPairs];
    const int P_all = M * topk;
    for (int i = threadIdx.x; i < P_all; i += blockDim.x) sid[i] = ids[i];
    for (int e = threadIdx.x; e < E; e += blockDim.x) R.cnt[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < P_all; i += blockDim.x) {
        const int t = i / topk, k = i - t * topk;
        const int e = sid[i];
        bool ok = e >= 0 && e < E;
        for (int j = 0; ok && j < k; ++j)
            if (sid[t * topk + j] == e) ok = false;
        R.valid[i] = ok ? 1 : 0;
        if (ok) atomicAdd(&R.cnt[e], 1);
        else if (blockIdx.x == 0) set_status(ws, DG_DEVERR_BAD_TOPK_ID);
    }
    __syncthreads();
    // Exclusive scans over the experts of (count > 0) and count, 32 experts per warp
    // chunk: chunk totals first, then each chunk's prefix from ballots (an expert's
    // count is at most M <= 16, so five bit planes give the count prefix) plus the
    // totals of the chunks before it.
    {
        __shared__ int tot_u[kMoeMaxE / 32], tot_p[kMoeMaxE / 32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
        const int chunks = (E + 31) / 32;
        const unsigned lt = (1u << lane) - 1u;
        for (int ch = warp; ch < chunks; ch += nw) {
            const int e = ch * 32 + lane;
            const int c = e < E ? R.cnt[e] : 0;
            const unsigned act = __ballot_sync(kFull, c > 0);
            const int sum = __reduce_add_sync(kFull, static_cast<unsigned>(c));
            if (lane == 0) {
                tot_u[ch] = __popc(act);
                tot_p[ch] = sum;
            }
        }
        __syncthreads();
        for (int ch = warp; ch < chunks; ch += nw) {
            int carry_u = 0, carry_p = 0;
            for (int j = 0; j < ch; ++j) {
                carry_u += tot_u[j];
                carry_p += tot_p[j];
            }
            const int e = ch * 32 + lane;
            const int c = e < E ? R.cnt[e] : 0;
            const unsigned act = __ballot_sync(kFull, c > 0);
            int ex_p = 0;
#pragma unroll
            for (int b = 0; b < 5; ++b) ex_p += __popc(__ballot_sync(kFull, (c >> b) & 1) & lt) << b;
            const int ex_u = carry_u + __popc(act & lt);
            ex_p += carry_p;
            if (e < E) {
                if (c > 0) {
                    R.experts[ex_u] = static_cast<int16_t>(e);
                    R.offs[ex_u] = static_cast<int16_t>(ex_p);
                }
                R.cnt[e] = ex_p;    // now the expert's first pair position
            }
            if (ch == chunks - 1 && lane == 31) {
                R.U = ex_u + (c > 0 ? 1 : 0);
                R.P = ex_p + c;
                R.offs[R.U] = static_cast<int16_t>(R.P);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < P_all; i += blockDim.x) {
        if (!R.valid[i]) continue;
        const int e = sid[i];
        int rank = 0;
        for (int j = 0; j < i; ++j)
            if (R.valid[j] && sid[j] == e) ++rank;
        const int pos = R.cnt[e] + rank;
        R.ptok[pos] = static_cast<int8_t>(i / topk);
        R.pslot[pos] = static_cast<int8_t>(i % topk);
    }
    for (int t = threadIdx.x; t < M; t += blockDim.x) {
        int n = 0;
        for (int k = 0; k < topk; ++k) n += R.valid[t * topk + k];
        R.nvalid[t] = n;
    }
    __syncthreads();
}

// Sense-reversing grid barrier for a grid whose CTAs are all resident at once (a
// persistent grid sized by the occupancy and launched cooperatively, so that no other
// kernel, of this stream or another, can keep one of them off an SM).
// Counter at bar[0], generation at bar[1]; the last arriver resets the counter for
// the next call.  One thread per CTA calls it.  Bounded: false after 2 s, or at
// once when `abort_flag` (if given) is raised.
__device__ inline bool grid_barrier(unsigned* bar, volatile int* abort_flag = nullptr)
{
    constexpr unsigned long long kLimitNs = 2000000000ull;
    volatile unsigned* gen = bar + 1;
    const unsigned my_gen = *gen;
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
        bar[0] = 0u;
        __threadfence();
        atomicAdd(bar + 1, 1u);
        return true;
    }
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t i = 1;; ++i) {
        if (*gen != my_gen) return true;
        if ((i & 63u) == 0) {
            if (abort_flag && *abort_flag) return false;
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (t - t0 > kLimitNs) return false;
        }
    }
}

}  // namespace dg
