// zero_step_table.cuh -- the template instances one 16-bit format needs.
// Rank counts with a compiled-in loop (1, 2, 4, 8, 16, 32, 64) get a fully
// unrolled fold; any other count uses the generic instance (ND = 0).
#pragma once

#include "zero_launch.h"
#include "zero_step_kernels.cuh"
#include "zero_tma.cuh"

namespace zero {

template <int DT, int ND>
static const void* fused_or_reduce(int kind)
{
    switch (kind) {
    case K_FUSED: return (const void*)k_fused<DT, ND>;
    case K_REDUCE_G32:
        if constexpr (ND == 0 || ND >= 4) return (const void*)k_reduce<DT, ND, true>;
        return nullptr;
    case K_REDUCE_ONLY:
        if constexpr (ND == 0 || ND < 4) return (const void*)k_reduce<DT, ND, false>;
        return nullptr;
    case K_UPDATE_RECOMPUTE:
        if constexpr (ND == 0 || ND < 4) return (const void*)k_update<DT, ND, true>;
        return nullptr;
    case K_UPDATE_G32:
        return (const void*)k_update<DT, 0, false>;
    default: return nullptr;
    }
}

// The qwZ-epilogue instances (ZeRO-3 steps that also quantize the updated
// shard) and the ping-pong step's passes, compiled in their own translation
// units.
template <int DT, int ND>
static const void* fused_or_update_q(int kind)
{
    switch (kind) {
    case K_FUSED_Q8: return (const void*)k_fused_q<DT, ND, 8>;
    case K_FUSED_Q4: return (const void*)k_fused_q<DT, ND, 4>;
    case K_UPDATE_G32_Q8: return (const void*)k_update<DT, 0, false, 8>;
    case K_UPDATE_G32_Q4: return (const void*)k_update<DT, 0, false, 4>;
    case K_UPDATE_RECOMPUTE_Q8:
        if constexpr (ND == 0 || ND < 4) return (const void*)k_update<DT, ND, true, 8>;
        return nullptr;
    case K_UPDATE_RECOMPUTE_Q4:
        if constexpr (ND == 0 || ND < 4) return (const void*)k_update<DT, ND, true, 4>;
        return nullptr;
    case K_FUSED_PP: return (const void*)k_fused_pp<DT, ND>;
    default: return nullptr;
    }
}

template <int DT>
static const void* step_kernel_q_dt(int kind, int nd)
{
    if (kind == K_PP_REPAIR) return (const void*)k_pp_repair<DT>;
    switch (nd) {
    case 1:  return fused_or_update_q<DT, 1>(kind);
    case 2:  return fused_or_update_q<DT, 2>(kind);
    case 4:  return fused_or_update_q<DT, 4>(kind);
    case 8:  return fused_or_update_q<DT, 8>(kind);
    case 16: return fused_or_update_q<DT, 16>(kind);
    case 32: return fused_or_update_q<DT, 32>(kind);
    case 64: return fused_or_update_q<DT, 64>(kind);
    default: return fused_or_update_q<DT, 0>(kind);
    }
}

template <int DT>
static const void* step_kernel_dt(int kind, int nd)
{
    if (kind == K_BUCKET_FINALIZE) return (const void*)k_bucket_finalize<DT>;
    if (kind == K_REDUCE_G32_TMA) {
        switch (nd) {
        case 4:  return (const void*)k_reduce_tma<DT, 4>;
        case 8:  return (const void*)k_reduce_tma<DT, 8>;
        case 16: return (const void*)k_reduce_tma<DT, 16>;
        case 32: return (const void*)k_reduce_tma<DT, 32>;
        default: return (const void*)k_reduce_tma<DT, 0>;
        }
    }
    switch (nd) {
    case 1:  return fused_or_reduce<DT, 1>(kind);
    case 2:  return fused_or_reduce<DT, 2>(kind);
    case 4:  return fused_or_reduce<DT, 4>(kind);
    case 8:  return fused_or_reduce<DT, 8>(kind);
    case 16: return fused_or_reduce<DT, 16>(kind);
    case 32: return fused_or_reduce<DT, 32>(kind);
    case 64: return fused_or_reduce<DT, 64>(kind);
    default: return fused_or_reduce<DT, 0>(kind);
    }
}

}  // namespace zero
