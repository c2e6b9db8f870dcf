// Instantiates the cluster-barrier exchange-and-add kernels for IEEE binary16.
#include "ar_allreduce_cluster.cuh"

namespace tda {
const void *allreduce_cluster_kernel_ptr_f16(int R, int sub, bool traced, bool paced) {
    return allreduce_cluster_ptr<F16Ops>(R, sub, traced, paced);
}
}  // namespace tda
