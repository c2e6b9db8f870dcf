// Instantiates the one-shot and tagged-word exchange-and-add kernels for bfloat16.
#include "ar_allreduce.cuh"

namespace tda {
const void *allreduce_kernel_ptr_bf16(int R, int U, bool fused, bool traced) {
    return allreduce_ptr<BF16Ops>(R, U, fused, traced);
}
}  // namespace tda
