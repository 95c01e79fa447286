// zero_step_q_fp16.cu -- fp16 step kernels with the qwZ quantizer in the
// update's epilogue (ZeRO-3 steps that also quantize the updated shard).
#include "zero_step_table.cuh"

namespace zero {
const void* step_kernel_q_fp16(int kind, int nd) { return step_kernel_q_dt<0>(kind, nd); }
}  // namespace zero
