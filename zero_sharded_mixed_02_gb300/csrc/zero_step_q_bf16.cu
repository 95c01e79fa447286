// zero_step_q_bf16.cu -- bf16 step kernels with the qwZ quantizer in the
// update's epilogue (ZeRO-3 steps that also quantize the updated shard).
#include "zero_step_table.cuh"

namespace zero {
const void* step_kernel_q_bf16(int kind, int nd) { return step_kernel_q_dt<1>(kind, nd); }
}  // namespace zero
