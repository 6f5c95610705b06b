// dg_a8.cu -- the A8W8 activation quantisation on its own (dg_quant_a8_blockscale):
// the same device code as the tensor-core A8W8 kernel's prologue, writing the codes
// and the per-(token, block) scales out.
#include "dg_a8.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

// Eight lanes per (token, block); grid covers M * ceil(K/128) blocks.
__global__ void __launch_bounds__(256) a8_quant_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ q,
                                                       float* __restrict__ sx, int M, int K)
{
    pdl_launch_dependents();
    pdl_wait();
    const int nb = (K + kA8Block - 1) / kA8Block;
    const long long p = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
    const int ch = threadIdx.x & 7;
    const bool ok = p < static_cast<long long>(M) * nb;
    const int t = ok ? static_cast<int>(p / nb) : 0;
    const int b = ok ? static_cast<int>(p - static_cast<long long>(t) * nb) : 0;
    const int k0 = b * kA8Block + ch * 16;
    float v[16];
    a8_load16(x + static_cast<size_t>(t) * K, ok ? k0 : K, K, v);
    const float amax = a8_block_amax(v);
    const float r = a8_recip_scale(amax);
    if (ok && k0 < K) *reinterpret_cast<uint4*>(q + static_cast<size_t>(t) * K + k0) = a8_codes(v, r);
    if (ok && ch == 0) sx[static_cast<size_t>(t) * nb + b] = a8_scale(amax);
}

}  // namespace

dg_status launch_a8_quant(const void* x, void* q, float* sx, int M, int K, cudaStream_t stream)
{
    const long long lanes = static_cast<long long>(M) * ((K + kA8Block - 1) / kA8Block) * 8;
    const unsigned grid = static_cast<unsigned>((lanes + 255) / 256);
    const uint16_t* xa = static_cast<const uint16_t*>(x);
    uint8_t* qa = static_cast<uint8_t*>(q);
    void* args[] = {&xa, &qa, &sx, &M, &K};
    if (launch_kernel(reinterpret_cast<const void*>(&a8_quant_kernel), grid, 256, 0, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg
