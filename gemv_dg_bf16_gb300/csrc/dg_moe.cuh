// dg_moe.cuh -- argument block and workspace layout of the MoE kernels.
#pragma once

#include <cstddef>
#include <cstdint>

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

}  // namespace dg
