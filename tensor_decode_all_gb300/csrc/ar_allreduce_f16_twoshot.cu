// Instantiates the two-shot exchange-and-add kernels for IEEE binary16.
#include "ar_allreduce.cuh"

namespace tda {
const void *allreduce_twoshot_kernel_ptr_f16(int R, int U, bool fused, bool traced) {
    return allreduce_twoshot_ptr_any<F16Ops>(R, U, fused, traced);
}
}  // namespace tda
