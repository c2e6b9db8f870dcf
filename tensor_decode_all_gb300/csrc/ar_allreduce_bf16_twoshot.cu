// Instantiates the two-shot exchange-and-add kernels for bfloat16.
#include "ar_allreduce.cuh"

namespace tda {
const void *allreduce_twoshot_kernel_ptr_bf16(int R, int U, bool fused, bool traced) {
    return allreduce_twoshot_ptr_any<BF16Ops>(R, U, fused, traced);
}
}  // namespace tda
