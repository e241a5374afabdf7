// prodigy.h -- hooks of the Prodigy step-size controller used by the group entry points.
#pragma once

#include "factored.h"

struct optim_group;

namespace lmo {
struct ProdigyAttach;
// Enqueues the group's Prodigy statistics for this step on `s` (after its gradient pointers are
// uploaded, before its factored kernels) and returns the device scalars those kernels must read.
int prodigy_step_begin(optim_group* g, const optim_factored_hparams_t* hp, cudaStream_t s,
                       const FactoredDevScalars** kdev);
// Releases the group's attachment (group destruction).
void prodigy_detach(optim_group* g);
}  // namespace lmo
