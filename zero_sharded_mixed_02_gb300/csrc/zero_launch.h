// zero_launch.h -- host-side interface between the plan code and the kernels.
#pragma once

#include <cuda_runtime.h>

#include "zero_common.cuh"

namespace zero {

enum Kind {
    K_REDUCE_G32 = 0,        // pass 1, writes the fp32 gradient      (nd >= 4)
    K_REDUCE_ONLY = 1,       // pass 1, flag + norm only              (nd < 4)
    K_UPDATE_G32 = 2,        // pass 2 from the fp32 gradient          (nd >= 4)
    K_UPDATE_RECOMPUTE = 3,  // pass 2 re-reading the 16-bit gradients (nd < 4)
    K_FUSED = 4,             // single pass (no clip, no dynamic scale)
    K_REDUCE_G32_TMA = 5,    // pass 1 with TMA bulk staging of the rank rows (runtime nd)
    K_BUCKET_FINALIZE = 6,   // bucketed step: norm and bookkeeping from the bucket partials
    // ZeRO-3 steps with the qwZ quantizer in the update's epilogue (8 or 4 bits)
    K_FUSED_Q8 = 7,
    K_FUSED_Q4 = 8,
    K_UPDATE_G32_Q8 = 9,
    K_UPDATE_G32_Q4 = 10,
    K_UPDATE_RECOMPUTE_Q8 = 11,
    K_UPDATE_RECOMPUTE_Q4 = 12,
    // ping-pong steps (zero_step_pingpong): the single pass and its repair pass
    K_FUSED_PP = 13,
    K_PP_REPAIR = 14
};

// Kernel function for (dtype, kind, nd); nullptr if that combination is not
// built (the plan never asks for one).
const void* step_kernel(int dtype, int kind, int nd);

const void* step_kernel_fp16(int kind, int nd);
const void* step_kernel_bf16(int kind, int nd);
const void* step_kernel_q_fp16(int kind, int nd);   // the K_*_Q* kinds
const void* step_kernel_q_bf16(int kind, int nd);

struct GatherArgs {
    const uint16_t* src[ZERO_MAX_ND];   // rank k's slice of the unit
    uint16_t* out;
    int64_t   len;                      // unit length
    int64_t   slice;                    // slice length (multiple of 64)
    int       nd;
};
cudaError_t launch_gather(const GatherArgs& a, int sms, cudaStream_t stream);

}  // namespace zero
