// factored.h -- plan and launcher of the factored second-moment step (Adafactor / Prodigy).
#pragma once

#include <vector>

#include "internal.h"

namespace lmo {

// The scalars of a Prodigy-mode step that depend on d, when d lives in device memory (written
// each step by the Prodigy statistics kernel before the factored kernels read it).
struct FactoredDevScalars {
    float alpha, lr_eff, nwdlr, unum;
};

// Per-step scalars (host-computed: double, then one rounding to fp32).  unum: the update's
// numerator factor (1 for Adafactor, d for Prodigy), applied to each element's update before its
// sum of squares and its clip, as the factored step defines it.  kdev (may be null): device copy
// of the d-dependent scalars, which then replace the host values.
struct FactoredScalars {
    float b2t, alpha, eps1, eps2, clip, lr_eff, nwdlr;
    int32_t mode;
    float unum;
    const FactoredDevScalars* kdev;
};

// The scalars of a step with hyper-parameters hp at step `step` with step size d (hp->d unless
// a Prodigy controller supplies it).
FactoredScalars factored_scalars(const optim_factored_hparams_t* hp, int64_t step, float d);

struct FactoredPlan;
int factored_plan_build(FactoredPlan*& plan, const std::vector<optim_tensor_desc_t>& desc);
void factored_plan_free(FactoredPlan*& plan);
// `nonfinite` (may be null): counter of update CTAs that stored a non-finite weight.
// `apply_wait` (may be null): an event that every update kernel of the step waits for (work
// that must read the weights before they change).
int launch_factored_step(const FactoredPlan* plan, const uint16_t* const* d_grads,
                         const FactoredScalars& k, cudaStream_t s, cudaEvent_t mid, unsigned long long* nonfinite,
                         cudaEvent_t apply_wait);

}  // namespace lmo
