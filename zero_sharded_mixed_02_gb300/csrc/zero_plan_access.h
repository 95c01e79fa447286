// zero_plan_access.h -- what the files beside zero_abi.cu may read or change of a
// plan (host code only; the plan itself is defined in zero_abi.cu).
#pragma once

#include <cstdint>
#include <vector>

#include "zero_b200.h"

namespace zero {

int plan_nd(zero_plan_t plan);
int plan_stage(zero_plan_t plan);
int plan_dtype(zero_plan_t plan);

// The layout of a plan: stages 0-2 one flat vector of nd * shard elements;
// stage 3 units, each cut into nd slices (unit_slice) placed at unit_off in a
// rank's shard.
struct PlanLayout {
    uint64_t psi = 0;
    int nd = 1, stage = 0, dtype = 0, device = 0;
    uint64_t shard = 0;                       // stages 0-2: S; stage 3: one rank's shard
    uint64_t model_hash = 0;                  // identity of the tensor shape list
    std::vector<uint64_t> unit_len, unit_slice, unit_off;
};
void plan_layout(zero_plan_t plan, PlanLayout* out);

// The optimizer scalars carried from step to step.
struct PlanScalars {
    float loss_scale;
    int32_t good_steps;
    int64_t t;
    double beta1_pow;
    double beta2_pow;
};
// Waits for the plan's last step, then reads them.
zero_status_t plan_scalars_get(zero_plan_t plan, PlanScalars* out);
// Replaces them (and resets the last-step report to its before-any-step state).
zero_status_t plan_scalars_set(zero_plan_t plan, const PlanScalars& sc);

// What the last step's reduce pass settled (waits for it).
struct PlanStepStatus {
    int skipped = 0, overflow = 0;
    double grad_norm = 0.0;
    float clip_coef = 1.0f, bc1 = 0.0f, bc2 = 0.0f, used_scale = 1.0f;
};
zero_status_t plan_step_status(zero_plan_t plan, PlanStepStatus* out);
void plan_hparams(zero_plan_t plan, zero_hparams_t* out);

// Launch `fn`, a reduce-pass kernel taking (StepArgs, uint16_t* g16), over the
// plan's gradients as the step's reduce pass (the grid of the plain reduce
// pass; the plan's step event recorded after it).
zero_status_t plan_launch_reduce16(zero_plan_t plan, const void* fn, const void* grads, void* g16,
                                   void* stream);

// A plan whose state a failed load left half-written refuses steps and gathers.
void plan_set_poisoned(zero_plan_t plan, bool poisoned);
bool plan_poisoned(zero_plan_t plan);

// Pinned host staging owned by the plan: `count` buffers of at least `bytes`
// each, allocated on first use and kept until the plan is destroyed.  NULL on
// allocation failure.
void* const* plan_staging(zero_plan_t plan, int count, uint64_t bytes);

}  // namespace zero
