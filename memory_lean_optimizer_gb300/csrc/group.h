// group.h -- the group handle behind optim_group_t (shared by api.cu and offload.cu).
#pragma once

#include <vector>

#include "factored.h"
#include "internal.h"

namespace lmo {
struct OffloadBinding;
struct ProdigyAttach;
// Bounded host wait: polls the event until it completes or `timeout_s` passes (OPTIM_ETIMEOUT).
int wait_event(cudaEvent_t ev, double timeout_s, const char* what);
constexpr double kWaitTimeout = 120.0;
}  // namespace lmo

struct optim_group {
    int32_t kind = 0;
    int device = 0;
    int32_t n = 0;
    std::vector<optim_tensor_desc_t> desc;
    // device tables
    lmo::TensorRec* d_tensors = nullptr;
    const uint16_t** d_grads = nullptr;
    lmo::ScaleRec* d_scales = nullptr;
    lmo::Chunk* d_chunks = nullptr;
    unsigned long long* d_nonfinite = nullptr;
    uint8_t* d_zero_chunk = nullptr;   // one flag per u16-state chunk, written by the pre-pass
    int32_t n_chunks_large = 0;
    int32_t n_chunks_total = 0;
    int64_t chunk = lmo::kChunk;       // elements per chunk of this group (set by kind at creation)
    lmo::FactoredPlan* fplan = nullptr;
    // gradient pointers: host copy of the last upload, two pinned staging slots
    std::vector<const void*> cur_grads;
    bool grads_valid = false;
    const void** h_stage[2] = {nullptr, nullptr};
    cudaEvent_t stage_ev[2] = {nullptr, nullptr};
    int stage_slot = 0;
    cudaEvent_t sync_ev = nullptr;
    // step bookkeeping
    int64_t last_step = 0;
    double mu_product = 1.0;
    int next_parity = 0;
    cudaStream_t last_stream = nullptr;
    cudaEvent_t profile_ev = nullptr;
    lmo::OffloadBinding* offload = nullptr;   // non-NULL: res/m/v are pinned host buffers
    lmo::ProdigyAttach* prodigy = nullptr;    // non-NULL: d comes from a Prodigy controller
    // one-launch steps (k_nadam_fused): the group's grid-barrier counter and its running total
    unsigned* d_bar = nullptr;
    unsigned bar_total = 0;
    // a NAdam step begun (pre-pass enqueued, or deferred into the one-launch step) and not yet ended
    bool pending = false;
    bool pending_fused = false;
    int64_t pending_step = 0;
    double pending_mu = 1.0;
    lmo::NadamScalars pending_k{};
    const lmo::TensorRec* pending_table = nullptr;
    cudaStream_t pending_stream = nullptr;
};

namespace lmo {
// Offload hooks used by the step entry point (offload.cu).  begin: make sure the group's states
// are (being) copied into a staging slot, make `compute` wait for that copy, and return the
// device tensor table that points into the slot.  end: enqueue the write-back after the kernels.
int offload_step_begin(optim_group* g, cudaStream_t compute, const TensorRec** table);
// OPTIM_EINVAL unless the group's device is current.
int check_group_device(const optim_group* g);
// Bounded wait for the work of the group's last step call.
int sync_group(optim_group* g);
int offload_step_end(optim_group* g, cudaStream_t compute);
void offload_unbind(optim_group* g);
}  // namespace lmo
