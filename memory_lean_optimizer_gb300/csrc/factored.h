// factored.h -- plan and launcher of the factored second-moment step (Adafactor / Prodigy).
#pragma once

#include <vector>

#include "internal.h"

namespace lmo {

// Per-step scalars (host-computed: double, then one rounding to fp32).
struct FactoredScalars {
    float b2t, alpha, eps1, eps2, clip, lr_eff, nwdlr;
    int32_t mode;
};

struct FactoredPlan;
int factored_plan_build(FactoredPlan*& plan, const std::vector<optim_tensor_desc_t>& desc);
void factored_plan_free(FactoredPlan*& plan);
// `nonfinite` (may be null): counter of update CTAs that stored a non-finite weight.
int launch_factored_step(const FactoredPlan* plan, const uint16_t* const* d_grads,
                         const FactoredScalars& k, cudaStream_t s, cudaEvent_t mid, unsigned long long* nonfinite);

}  // namespace lmo
