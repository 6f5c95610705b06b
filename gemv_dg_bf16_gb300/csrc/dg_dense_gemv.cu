// Instantiations of the dense CUDA-core family for the bf16 linear.
#include "dg_cc_dense.cuh"
#include "dg_dense_table.cuh"

namespace dg {
const void* dense_kernel_gemv(int mt, int R, bool ksplit) { return dense_lookup<WT_BF16, EPI_STORE>(mt, R, ksplit); }
const void* bulk_kernel_gemv(int mt) { return bulk_lookup<WT_BF16, EPI_STORE>(mt); }
}  // namespace dg
