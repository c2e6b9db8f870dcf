// Instantiates the one-shot and tagged-word exchange-and-add kernels for IEEE binary16.
#include "ar_allreduce.cuh"

namespace tda {
const void *allreduce_kernel_ptr_f16(int R, int U, bool fused, bool traced) {
    return allreduce_ptr<F16Ops>(R, U, fused, traced);
}
}  // namespace tda
