// zero_step_bf16.cu -- step kernels for bf16 gradients and parameters.
#include "zero_step_table.cuh"

namespace zero {
const void* step_kernel_bf16(int kind, int nd) { return step_kernel_dt<1>(kind, nd); }
}  // namespace zero
