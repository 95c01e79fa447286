// zero_step_fp16.cu -- step kernels for fp16 gradients and parameters.
#include "zero_step_table.cuh"

namespace zero {
const void* step_kernel_fp16(int kind, int nd) { return step_kernel_dt<0>(kind, nd); }
}  // namespace zero
