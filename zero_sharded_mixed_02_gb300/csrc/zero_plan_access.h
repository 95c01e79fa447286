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

// A plan whose state a failed load left half-written refuses steps and gathers.
void plan_set_poisoned(zero_plan_t plan, bool poisoned);
bool plan_poisoned(zero_plan_t plan);

// Pinned host staging owned by the plan: `count` buffers of at least `bytes`
// each, allocated on first use and kept until the plan is destroyed.  NULL on
// allocation failure.
void* const* plan_staging(zero_plan_t plan, int count, uint64_t bytes);

}  // namespace zero
