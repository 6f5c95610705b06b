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

// Every CTA computes the same routing tables (deterministic, no atomics on order).
// topk_ids is read from global memory once, into shared memory.
__device__ inline void route_scan(Route& R, const int32_t* __restrict__ ids, int M, int topk, int E,
                           uint8_t* ws)
{
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
    // Warp 0: exclusive scans over experts of (count > 0) and count.
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry_u = 0, carry_p = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? R.cnt[e] : 0;
            const int a = c > 0 ? 1 : 0;
            int su = a, sp = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int nu = __shfl_up_sync(kFull, su, o);
                const int np = __shfl_up_sync(kFull, sp, o);
                if (lane >= o) {
                    su += nu;
                    sp += np;
                }
            }
            const int ex_u = carry_u + su - a, ex_p = carry_p + sp - c;
            if (e < E) {
                if (a) {
                    R.experts[ex_u] = static_cast<int16_t>(e);
                    R.offs[ex_u] = static_cast<int16_t>(ex_p);
                }
                R.cnt[e] = ex_p;    // now the expert's first pair position
            }
            carry_u += __shfl_sync(kFull, su, 31);
            carry_p += __shfl_sync(kFull, sp, 31);
        }
        if (lane == 0) {
            R.U = carry_u;
            R.P = carry_p;
            R.offs[carry_u] = static_cast<int16_t>(carry_p);
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

}  // namespace dg
