// Instantiations of the dense CUDA-core family for the fp8 head + greedy argmax.
#include "dg_cc_dense.cuh"
#include "dg_dense_table.cuh"

namespace dg {
const void* dense_kernel_head(int mt, int R, bool ksplit) { return dense_lookup<WT_E4M3, EPI_HEAD>(mt, R, ksplit); }
const void* bulk_kernel_head(int mt) { return bulk_lookup<WT_E4M3, EPI_HEAD>(mt); }
}  // namespace dg
