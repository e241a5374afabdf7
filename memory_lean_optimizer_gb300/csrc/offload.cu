// offload.cu -- pinned-host offload of Kahan residuals and moment codes between steps.
//
// The pages keep AdamW's two moments and the Kahan residuals in CPU memory between steps,
// moving each parameter group's states to the GPU for its update and back afterwards ("Amazing
// Flux FFT quality on a 5090", sd-scripts PR #2187, first post; "Kahan summation for
// Adafactor-optimized Flux FFT", sd-scripts PR #2159, PR description).  Here the states of an
// offloaded group live in pinned host memory; an engine owns a ring of device staging slots, an
// H2D and a D2H copy stream, and per-slot events, so that the copy-in of group k+1 and the
// copy-out of group k-1 overlap the update kernels of group k:
//
//   prefetch(g):  h2d  waits slot.d2h_done   -> H2D copies -> record slot.h2d_done
//   step(g):      comp waits slot.h2d_done   -> K1, K2 on the slot's tensor table
//                                            -> record slot.comp_done
//                 d2h  waits slot.comp_done  -> D2H copies -> record slot.d2h_done
//
// Every dependency is a device-side event wait; the host never blocks in a step.  Weights and
// gradients stay on the device; per-tensor scale records (64 bytes per tensor) stay on the device.
// Host fault injection for tests: LMOPT_FAULT_INJECT=h2d | d2h | alloc makes the corresponding
// call fail with OPTIM_ECUDA / OPTIM_ENOMEM before it enqueues anything.
#include <cstdlib>
#include <cstring>
#include <vector>

#include "group.h"

namespace lmo {

struct Slot {
    char* base = nullptr;
    cudaEvent_t h2d_done = nullptr, comp_done = nullptr, d2h_done = nullptr;
    optim_group* owner = nullptr;   // group prefetched into this slot and not yet stepped
};

}  // namespace lmo

struct optim_offload {
    int device = 0;
    size_t slot_bytes = 0;
    std::vector<lmo::Slot> slots;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t sync_ev = nullptr;
    uint64_t next = 0;
    int bound = 0;
    uint64_t bytes_h2d = 0, bytes_d2h = 0;
};

namespace lmo {

struct OffloadBinding {
    optim_offload* eng = nullptr;
    std::vector<size_t> off_res, off_m, off_v, sz_m;   // per tensor, within a slot
    size_t need = 0;
    TensorRec* d_tables = nullptr;                     // n_slots tables of n records
    int slot = -1;                                     // slot holding the prefetched states
};

static bool fault(const char* what) {
    const char* f = std::getenv("LMOPT_FAULT_INJECT");
    return f && std::strcmp(f, what) == 0;
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static int prefetch(optim_group* g) {
    OffloadBinding* b = g->offload;
    optim_offload* e = b->eng;
    if (b->slot >= 0) return OPTIM_OK;
    const int s = (int)(e->next % e->slots.size());
    Slot& sl = e->slots[s];
    if (sl.owner != nullptr)
        return set_error(OPTIM_ESTATE, "no free staging slot: step the groups already prefetched first");
    if (fault("h2d")) return set_error(OPTIM_ECUDA, "injected H2D copy failure");
    int rc = check_cuda(cudaStreamWaitEvent(e->h2d, sl.d2h_done, 0), "offload h2d wait");
    for (int32_t i = 0; i < g->n && !rc; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        if (d.numel == 0) continue;
        if (d.res_u16)
            rc = check_cuda(cudaMemcpyAsync(sl.base + b->off_res[i], d.res_u16, 2 * d.numel, cudaMemcpyHostToDevice, e->h2d), "offload h2d");
        if (!rc) rc = check_cuda(cudaMemcpyAsync(sl.base + b->off_m[i], d.m, b->sz_m[i], cudaMemcpyHostToDevice, e->h2d), "offload h2d");
        if (!rc) rc = check_cuda(cudaMemcpyAsync(sl.base + b->off_v[i], d.v, b->sz_m[i], cudaMemcpyHostToDevice, e->h2d), "offload h2d");
        e->bytes_h2d += (d.res_u16 ? 2 * d.numel : 0) + 2 * b->sz_m[i];
    }
    if (!rc) rc = check_cuda(cudaEventRecord(sl.h2d_done, e->h2d), "offload h2d event");
    if (rc) return rc;
    sl.owner = g;
    b->slot = s;
    e->next++;
    return OPTIM_OK;
}

int offload_step_begin(optim_group* g, cudaStream_t compute, const TensorRec** table) {
    int rc = prefetch(g);
    if (rc) return rc;
    OffloadBinding* b = g->offload;
    if (fault("d2h")) return set_error(OPTIM_ECUDA, "injected D2H copy failure");
    Slot& sl = b->eng->slots[b->slot];
    rc = check_cuda(cudaStreamWaitEvent(compute, sl.h2d_done, 0), "offload compute wait");
    if (rc) return rc;
    *table = b->d_tables + (size_t)b->slot * g->n;
    return OPTIM_OK;
}

int offload_step_end(optim_group* g, cudaStream_t compute) {
    OffloadBinding* b = g->offload;
    optim_offload* e = b->eng;
    Slot& sl = e->slots[b->slot];
    int rc = check_cuda(cudaEventRecord(sl.comp_done, compute), "offload compute event");
    if (!rc) rc = check_cuda(cudaStreamWaitEvent(e->d2h, sl.comp_done, 0), "offload d2h wait");
    for (int32_t i = 0; i < g->n && !rc; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        if (d.numel == 0) continue;
        if (d.res_u16)
            rc = check_cuda(cudaMemcpyAsync(d.res_u16, sl.base + b->off_res[i], 2 * d.numel, cudaMemcpyDeviceToHost, e->d2h), "offload d2h");
        if (!rc) rc = check_cuda(cudaMemcpyAsync(d.m, sl.base + b->off_m[i], b->sz_m[i], cudaMemcpyDeviceToHost, e->d2h), "offload d2h");
        if (!rc) rc = check_cuda(cudaMemcpyAsync(d.v, sl.base + b->off_v[i], b->sz_m[i], cudaMemcpyDeviceToHost, e->d2h), "offload d2h");
        e->bytes_d2h += (d.res_u16 ? 2 * d.numel : 0) + 2 * b->sz_m[i];
    }
    if (!rc) rc = check_cuda(cudaEventRecord(sl.d2h_done, e->d2h), "offload d2h event");
    sl.owner = nullptr;
    b->slot = -1;
    return rc;
}

void offload_unbind(optim_group* g) {
    if (!g->offload) return;
    OffloadBinding* b = g->offload;
    if (b->slot >= 0) b->eng->slots[b->slot].owner = nullptr;
    b->eng->bound--;
    cudaFree(b->d_tables);
    delete b;
    g->offload = nullptr;
}

static int stream_wait_all(optim_offload* e) {
    for (cudaStream_t s : {e->h2d, e->d2h}) {
        int rc = check_cuda(cudaEventRecord(e->sync_ev, s), "offload sync event");
        if (!rc) rc = wait_event(e->sync_ev, kWaitTimeout, "offload copy stream");
        if (rc) return rc;
    }
    return OPTIM_OK;
}

static void engine_free(optim_offload* e) {
    for (Slot& s : e->slots) {
        cudaFree(s.base);
        if (s.h2d_done) cudaEventDestroy(s.h2d_done);
        if (s.comp_done) cudaEventDestroy(s.comp_done);
        if (s.d2h_done) cudaEventDestroy(s.d2h_done);
    }
    if (e->sync_ev) cudaEventDestroy(e->sync_ev);
    if (e->h2d) cudaStreamDestroy(e->h2d);
    if (e->d2h) cudaStreamDestroy(e->d2h);
    delete e;
}

}  // namespace lmo

using namespace lmo;

extern "C" {

int optim_offload_create(size_t slot_bytes, int32_t n_slots, optim_offload_t** out) {
    if (!out || slot_bytes == 0 || n_slots < 2 || n_slots > 64)
        return set_error(OPTIM_EINVAL, "need out, slot_bytes > 0 and 2 <= n_slots <= 64");
    *out = nullptr;
    if (fault("alloc")) return set_error(OPTIM_ENOMEM, "injected staging allocation failure");
    optim_offload* e = new optim_offload();
    e->slot_bytes = slot_bytes;
    e->slots.resize(n_slots);
    int rc = check_cuda(cudaGetDevice(&e->device), "cudaGetDevice");
    for (int s = 0; s < n_slots && !rc; ++s) {
        if (cudaMalloc(reinterpret_cast<void**>(&e->slots[s].base), slot_bytes) != cudaSuccess) {
            cudaGetLastError();
            rc = set_error(OPTIM_ENOMEM, "staging slot allocation of %zu bytes failed", slot_bytes);
            break;
        }
        rc = check_cuda(cudaEventCreateWithFlags(&e->slots[s].h2d_done, cudaEventDisableTiming), "event");
        if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&e->slots[s].comp_done, cudaEventDisableTiming), "event");
        if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&e->slots[s].d2h_done, cudaEventDisableTiming), "event");
    }
    if (!rc) rc = check_cuda(cudaStreamCreateWithFlags(&e->h2d, cudaStreamNonBlocking), "stream");
    if (!rc) rc = check_cuda(cudaStreamCreateWithFlags(&e->d2h, cudaStreamNonBlocking), "stream");
    if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&e->sync_ev, cudaEventDisableTiming), "event");
    if (rc) {
        engine_free(e);
        return rc;
    }
    *out = e;
    return OPTIM_OK;
}

int optim_offload_destroy(optim_offload_t* e) {
    if (!e) return set_error(OPTIM_EINVAL, "engine is NULL");
    if (e->bound > 0) return set_error(OPTIM_ESTATE, "%d groups are still attached", e->bound);
    int rc = stream_wait_all(e);
    engine_free(e);
    return rc;
}

int optim_group_attach_offload(optim_group_t* g, optim_offload_t* e) {
    if (!g || !e) return set_error(OPTIM_EINVAL, "group or engine is NULL");
    if (g->kind != OPTIM_KIND_NADAM) return set_error(OPTIM_EINVAL, "only NADAM groups with u16 moments can be offloaded");
    if (g->offload) return set_error(OPTIM_ESTATE, "group already attached");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    if (g->device != e->device) return set_error(OPTIM_EINVAL, "group and engine are on different devices");
    OffloadBinding* b = new OffloadBinding();
    b->eng = e;
    size_t off = 0;
    for (int32_t i = 0; i < g->n; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        const size_t n = (size_t)d.numel;
        const size_t sm = (d.numel <= kSmall ? 4 : 2) * n;
        for (void* p : {d.res_u16, d.m, d.v}) {
            if (!p || n == 0) continue;
            cudaPointerAttributes a{};
            if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
                cudaGetLastError();
                delete b;
                return set_error(OPTIM_EINVAL, "tensor %d: state pointer is not known to CUDA (use pinned host memory)", i);
            }
            if (a.type != cudaMemoryTypeHost) {
                delete b;
                return set_error(OPTIM_EINVAL, "tensor %d: offloaded states must be pinned host memory", i);
            }
        }
        b->off_res.push_back(off);
        off += d.res_u16 ? round256(2 * n) : 0;
        b->off_m.push_back(off);
        off += round256(sm);
        b->off_v.push_back(off);
        off += round256(sm);
        b->sz_m.push_back(sm);
    }
    b->need = off;
    if (off > e->slot_bytes) {
        delete b;
        return set_error(OPTIM_EINVAL, "group needs %zu staging bytes, slots hold %zu", off, e->slot_bytes);
    }
    std::vector<TensorRec> tables((size_t)g->n * e->slots.size());
    for (size_t s = 0; s < e->slots.size(); ++s) {
        for (int32_t i = 0; i < g->n; ++i) {
            const optim_tensor_desc_t& d = g->desc[i];
            TensorRec& r = tables[s * g->n + i];
            r.w = static_cast<uint16_t*>(d.w_bf16);
            r.res = d.res_u16 ? reinterpret_cast<uint16_t*>(e->slots[s].base + b->off_res[i]) : nullptr;
            r.m = e->slots[s].base + b->off_m[i];
            r.v = e->slots[s].base + b->off_v[i];
            r.numel = d.numel;
            r.flags = (d.numel <= kSmall ? kFlagSmall : 0) | (d.res_u16 ? kFlagRes : 0);
            r.pad = 0;
        }
    }
    int rc = OPTIM_OK;
    if (cudaMalloc(reinterpret_cast<void**>(&b->d_tables), tables.size() * sizeof(TensorRec)) != cudaSuccess) {
        cudaGetLastError();
        rc = set_error(OPTIM_ENOMEM, "offload table allocation failed");
    }
    if (!rc) rc = check_cuda(cudaMemcpy(b->d_tables, tables.data(), tables.size() * sizeof(TensorRec), cudaMemcpyHostToDevice), "offload table upload");
    if (rc) {
        cudaFree(b->d_tables);
        delete b;
        return rc;
    }
    g->offload = b;
    e->bound++;
    return OPTIM_OK;
}

int optim_offload_prefetch(optim_group_t* g) {
    if (!g || !g->offload) return set_error(OPTIM_EINVAL, "group is NULL or not offloaded");
    return prefetch(g);
}

int optim_offload_sync(optim_offload_t* e, uint64_t* bytes_h2d, uint64_t* bytes_d2h) {
    if (!e) return set_error(OPTIM_EINVAL, "engine is NULL");
    int rc = stream_wait_all(e);
    if (bytes_h2d) *bytes_h2d = e->bytes_h2d;
    if (bytes_d2h) *bytes_d2h = e->bytes_d2h;
    return rc;
}

}  // extern "C"
