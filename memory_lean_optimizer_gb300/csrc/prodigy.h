// prodigy.h -- hooks of the Prodigy step-size controller used by the group entry points.
#pragma once

#include "factored.h"

struct optim_group;

namespace lmo {
struct ProdigyAttach;
// Enqueues the group's Prodigy work for this step (after its gradient pointers are uploaded,
// before its factored kernels): the d-dependent scalars on `s`, returned in *kdev for the
// factored kernels; the statistics on the group's own stream, concurrent with the factored
// kernels up to their update, which must wait for *done (the statistics read the weights).
int prodigy_step_begin(optim_group* g, const optim_factored_hparams_t* hp, cudaStream_t s,
                       const FactoredDevScalars** kdev, cudaEvent_t* done);
// Makes `s` wait for the statistics of the group's last step (end of a group call).
int prodigy_step_join(optim_group* g, cudaStream_t s);
// Releases the group's attachment (group destruction).
void prodigy_detach(optim_group* g);
}  // namespace lmo
