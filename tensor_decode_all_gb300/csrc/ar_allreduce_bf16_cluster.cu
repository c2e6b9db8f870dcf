// Instantiates the cluster-barrier exchange-and-add kernels for bfloat16.
#include "ar_allreduce_cluster.cuh"

namespace tda {
const void *allreduce_cluster_kernel_ptr_bf16(int R, int sub, bool traced, bool paced) {
    return allreduce_cluster_ptr<BF16Ops>(R, sub, traced, paced);
}
}  // namespace tda
