// Instantiations of the dense CUDA-core family for the fused gate/up + SiLU.mul.
#include "dg_cc_dense.cuh"
#include "dg_dense_table.cuh"

namespace dg {
const void* dense_kernel_gateup(int mt, int R, bool ksplit) { return dense_lookup<WT_BF16, EPI_GATEUP>(mt, R, ksplit); }
const void* bulk_kernel_gateup(int mt) { return bulk_lookup<WT_BF16, EPI_GATEUP>(mt); }
}  // namespace dg
