// offload.cu -- pinned-host offload of Kahan residuals and optimizer states between steps.
//
// The pages keep the optimizer states and the Kahan residuals in CPU memory between steps,
// moving each parameter group's states to the GPU for its update and back afterwards ("Amazing
// Flux FFT quality on a 5090", sd-scripts PR #2187, first post, and its fourth post for Adan;
// "Kahan summation for Adafactor-optimized Flux FFT", sd-scripts PR #2159, PR description).
// Here the states of an offloaded group live in pinned host memory; an engine owns a ring of
// device staging slots, an H2D and a D2H copy stream, and per-slot events, so that the copy-in
// of group k+1 and the copy-out of group k-1 overlap the update kernels of group k:
//
//   prefetch(g):  copy stream waits slot.d2h_done -> H2D copies -> record slot.h2d_done
//   step(g):      compute waits slot.h2d_done     -> kernels on the slot's tensor table
//                                                 -> record slot.comp_done
//   write-back(g): copy stream waits slot.comp_done -> D2H copies -> record slot.d2h_done
//
// Every dependency is a device-side event wait; the host never blocks in a step.  Weights,
// gradients and per-tensor scale records stay on the device.
//
// Two ways to attach a group:
//  - optim_group_attach_offload(group, engine): the group's descriptors point at pinned host
//    buffers; the copies go state by state, the step enqueues the write-back itself.
//  - optim_group_attach_host(group, image, bytes): the caller hands over one pinned buffer, the
//    group's packed host image (layout from optim_offload_layout, the same as a staging slot's,
//    so that each copy is a single transfer); the caller enqueues prefetch and write-back on
//    copy streams of its choice.  The staging ring is the library's own, one per device, grown
//    to the largest attached group.
// Host fault injection for tests: LMOPT_FAULT_INJECT=h2d | d2h | alloc makes the corresponding
// call fail with OPTIM_ECUDA / OPTIM_ENOMEM before it enqueues anything (and =timeout makes
// every bounded host wait of the library run out at once).
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "group.h"

namespace lmo {

struct Slot {
    char* base = nullptr;
    cudaEvent_t h2d_done = nullptr, comp_done = nullptr, d2h_done = nullptr;
    optim_group* owner = nullptr;   // group whose states are in this slot (prefetched, not yet written back)
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
    bool library_owned = false;               // the per-device ring of optim_group_attach_host
    std::vector<optim_group*> groups;         // groups attached to a library-owned ring
    uint64_t bytes_h2d = 0, bytes_d2h = 0;
};

namespace lmo {

// One host <-> slot transfer of a group: `host` bytes at slot offset `off`.
struct Region {
    size_t off;
    size_t bytes;
    char* host;
};

struct OffloadBinding {
    optim_offload* eng = nullptr;
    std::vector<size_t> off_res, off_m, off_v;          // per tensor, within a slot (and the image)
    std::vector<size_t> sz_res, sz_m, sz_v;
    std::vector<Region> regions;
    size_t need = 0;
    TensorRec* d_tables = nullptr;                      // n_slots tables of n records
    int slot = -1;                                      // slot holding the group's states
    bool image = false;                                 // attached with optim_group_attach_host
    bool stepped = false;                               // a step ran on the slot since prefetch
};

static bool fault(const char* what) { return fault_injected(what); }

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
static size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

// Bytes of a tensor's offloaded states: residual, m buffer, v buffer (layouts of lmopt.h).
static void state_bytes(int32_t kind, const optim_tensor_desc_t& d, size_t& res, size_t& m, size_t& v) {
    const size_t n = (size_t)d.numel;
    const bool small = d.numel <= kSmall;
    res = d.res_u16 ? 2 * n : 0;
    const size_t f24 = round16(2 * n) + n;
    switch (kind) {
    case OPTIM_KIND_NADAM: m = v = (small ? 4 : 2) * n; break;
    case OPTIM_KIND_NADAM_F24: m = v = small ? 4 * n : f24; break;
    case OPTIM_KIND_ADAN: m = 12 * ((n + 3) & ~size_t(3)); v = 2 * n; break;
    default: /* ADAN_F24 */ m = small ? 12 * ((n + 3) & ~size_t(3)) : 3 * round16(f24); v = 2 * n; break;
    }
    if (n == 0) res = m = v = 0;
}

static bool offloadable(int32_t kind) {
    return kind == OPTIM_KIND_NADAM || kind == OPTIM_KIND_NADAM_F24 || kind == OPTIM_KIND_ADAN ||
           kind == OPTIM_KIND_ADAN_F24;
}

// Slot (and image) layout of a group: per tensor residual, m, v, each at a 256-byte boundary.
static OffloadBinding* plan_binding(const optim_group* g) {
    OffloadBinding* b = new OffloadBinding();
    size_t off = 0;
    for (int32_t i = 0; i < g->n; ++i) {
        size_t r, m, v;
        state_bytes(g->kind, g->desc[i], r, m, v);
        b->sz_res.push_back(r);
        b->sz_m.push_back(m);
        b->sz_v.push_back(v);
        b->off_res.push_back(off);
        off += round256(r);
        b->off_m.push_back(off);
        off += round256(m);
        b->off_v.push_back(off);
        off += round256(v);
    }
    b->need = off;
    return b;
}

// Device tensor tables pointing into each slot of the binding's engine.
static int upload_tables(optim_group* g, OffloadBinding* b) {
    optim_offload* e = b->eng;
    std::vector<TensorRec> tables((size_t)g->n * e->slots.size());
    for (size_t s = 0; s < e->slots.size(); ++s) {
        for (int32_t i = 0; i < g->n; ++i) {
            const optim_tensor_desc_t& d = g->desc[i];
            TensorRec& r = tables[s * g->n + i];
            char* base = e->slots[s].base;
            r.w = static_cast<uint16_t*>(d.w_bf16);
            r.res = d.res_u16 ? reinterpret_cast<uint16_t*>(base + b->off_res[i]) : nullptr;
            r.m = base + b->off_m[i];
            r.v = base + b->off_v[i];
            r.numel = d.numel;
            r.flags = (d.numel <= kSmall ? kFlagSmall : 0) | (d.res_u16 ? kFlagRes : 0);
            r.pad = 0;
        }
    }
    if (!b->d_tables && cudaMalloc(reinterpret_cast<void**>(&b->d_tables), tables.size() * sizeof(TensorRec)) != cudaSuccess) {
        cudaGetLastError();
        b->d_tables = nullptr;
        return set_error(OPTIM_ENOMEM, "offload table allocation failed");
    }
    return check_cuda(cudaMemcpy(b->d_tables, tables.data(), tables.size() * sizeof(TensorRec), cudaMemcpyHostToDevice),
                      "offload table upload");
}

static int prefetch(optim_group* g, cudaStream_t copy) {
    OffloadBinding* b = g->offload;
    optim_offload* e = b->eng;
    if (b->slot >= 0) return OPTIM_OK;
    // the first free slot from the ring's cursor on (its previous write-back is waited for below)
    const int n_slots = (int)e->slots.size();
    int s = -1;
    for (int i = 0; i < n_slots && s < 0; ++i) {
        const int c = (int)((e->next + i) % n_slots);
        if (e->slots[c].owner == nullptr) s = c;
    }
    if (s < 0)
        return set_error(OPTIM_ESTATE, "no free staging slot: step (and write back) the groups already prefetched first");
    Slot& sl = e->slots[s];
    if (fault("h2d")) return set_error(OPTIM_ECUDA, "injected H2D copy failure");
    cudaStream_t cs = copy ? copy : e->h2d;
    int rc = check_cuda(cudaStreamWaitEvent(cs, sl.d2h_done, 0), "offload h2d wait");
    uint64_t bytes = 0;
    for (const Region& r : b->regions) {
        if (rc) break;
        if (r.bytes == 0) continue;
        rc = check_cuda(cudaMemcpyAsync(sl.base + r.off, r.host, r.bytes, cudaMemcpyHostToDevice, cs), "offload h2d");
        bytes += r.bytes;
    }
    if (!rc) rc = check_cuda(cudaEventRecord(sl.h2d_done, cs), "offload h2d event");
    if (rc) return rc;
    e->bytes_h2d += bytes;
    sl.owner = g;
    b->slot = s;
    b->stepped = false;
    e->next = (uint64_t)s + 1;
    return OPTIM_OK;
}

static int writeback(optim_group* g, cudaStream_t copy) {
    OffloadBinding* b = g->offload;
    optim_offload* e = b->eng;
    Slot& sl = e->slots[b->slot];
    cudaStream_t cs = copy ? copy : e->d2h;
    int rc = check_cuda(cudaStreamWaitEvent(cs, b->stepped ? sl.comp_done : sl.h2d_done, 0), "offload d2h wait");
    uint64_t bytes = 0;
    for (const Region& r : b->regions) {
        if (rc) break;
        if (r.bytes == 0) continue;
        rc = check_cuda(cudaMemcpyAsync(r.host, sl.base + r.off, r.bytes, cudaMemcpyDeviceToHost, cs), "offload d2h");
        bytes += r.bytes;
    }
    if (!rc) rc = check_cuda(cudaEventRecord(sl.d2h_done, cs), "offload d2h event");
    e->bytes_d2h += bytes;
    sl.owner = nullptr;
    b->slot = -1;
    b->stepped = false;
    return rc;
}

int offload_step_begin(optim_group* g, cudaStream_t compute, const TensorRec** table) {
    OffloadBinding* b = g->offload;
    if (b->image && b->slot < 0)
        return set_error(OPTIM_ESTATE, "group attached with optim_group_attach_host: call optim_offload_prefetch first");
    int rc = prefetch(g, nullptr);
    if (rc) return rc;
    if (fault("d2h")) return set_error(OPTIM_ECUDA, "injected D2H copy failure");
    Slot& sl = b->eng->slots[b->slot];
    rc = check_cuda(cudaStreamWaitEvent(compute, sl.h2d_done, 0), "offload compute wait");
    if (rc) return rc;
    *table = b->d_tables + (size_t)b->slot * g->n;
    return OPTIM_OK;
}

int offload_step_end(optim_group* g, cudaStream_t compute) {
    OffloadBinding* b = g->offload;
    Slot& sl = b->eng->slots[b->slot];
    int rc = check_cuda(cudaEventRecord(sl.comp_done, compute), "offload compute event");
    if (rc) return rc;
    b->stepped = true;
    if (b->image) return OPTIM_OK;            // the caller writes back
    return writeback(g, nullptr);
}

static int stream_wait_all(optim_offload* e) {
    for (cudaStream_t s : {e->h2d, e->d2h}) {
        int rc = check_cuda(cudaEventRecord(e->sync_ev, s), "offload sync event");
        if (!rc) rc = wait_event(e->sync_ev, kWaitTimeout, "offload copy stream");
        if (rc) return rc;
    }
    return OPTIM_OK;
}

static void free_slots(optim_offload* e) {
    for (Slot& s : e->slots) {
        cudaFree(s.base);
        s.base = nullptr;
    }
}

static int alloc_slots(optim_offload* e, size_t slot_bytes) {
    e->slot_bytes = slot_bytes;
    for (Slot& s : e->slots) {
        if (cudaMalloc(reinterpret_cast<void**>(&s.base), slot_bytes) != cudaSuccess) {
            cudaGetLastError();
            s.base = nullptr;
            return set_error(OPTIM_ENOMEM, "staging slot allocation of %zu bytes failed", slot_bytes);
        }
    }
    return OPTIM_OK;
}

static void engine_free(optim_offload* e) {
    free_slots(e);
    for (Slot& s : e->slots) {
        if (s.h2d_done) cudaEventDestroy(s.h2d_done);
        if (s.comp_done) cudaEventDestroy(s.comp_done);
        if (s.d2h_done) cudaEventDestroy(s.d2h_done);
    }
    if (e->sync_ev) cudaEventDestroy(e->sync_ev);
    if (e->h2d) cudaStreamDestroy(e->h2d);
    if (e->d2h) cudaStreamDestroy(e->d2h);
    delete e;
}

static int engine_new(size_t slot_bytes, int32_t n_slots, optim_offload** out) {
    *out = nullptr;
    if (fault("alloc")) return set_error(OPTIM_ENOMEM, "injected staging allocation failure");
    optim_offload* e = new optim_offload();
    e->slots.resize(n_slots);
    int rc = check_cuda(cudaGetDevice(&e->device), "cudaGetDevice");
    if (!rc) rc = alloc_slots(e, slot_bytes);
    for (int s = 0; s < n_slots && !rc; ++s) {
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

// The library's own staging ring of each device, for groups attached with
// optim_group_attach_host: three slots, grown (between steps, with no slot in use) to the
// largest attached group, freed when its last group goes.
constexpr int kMaxDevices = 64;
constexpr int32_t kLibrarySlots = 3;
static optim_offload* g_ring[kMaxDevices] = {nullptr};
static std::mutex g_ring_mu;

static int ring_bind(optim_group* g, OffloadBinding* b) {
    std::lock_guard<std::mutex> lock(g_ring_mu);
    if (g->device < 0 || g->device >= kMaxDevices) return set_error(OPTIM_EINVAL, "device %d out of range", g->device);
    optim_offload*& e = g_ring[g->device];
    int rc = OPTIM_OK;
    if (!e) {
        rc = engine_new(b->need, kLibrarySlots, &e);
        if (rc) return rc;
        e->library_owned = true;
    } else if (b->need > e->slot_bytes) {
        for (const Slot& s : e->slots)
            if (s.owner) return set_error(OPTIM_ESTATE, "the staging ring must grow, but a group's states are on the device: write them back first");
        // copies and kernels queued earlier may still use the old slots (also on callers' copy
        // streams): wait, bounded, for every slot's last events
        rc = stream_wait_all(e);
        for (Slot& s : e->slots)
            for (cudaEvent_t ev : {s.h2d_done, s.comp_done, s.d2h_done})
                if (!rc) rc = wait_event(ev, kWaitTimeout, "staging slot before resize");
        if (rc) return rc;
        free_slots(e);
        rc = alloc_slots(e, b->need);
        for (optim_group* o : e->groups)
            if (!rc) rc = upload_tables(o, o->offload);
        if (rc) return rc;
    }
    b->eng = e;
    rc = upload_tables(g, b);
    if (rc) {
        if (e->bound == 0) {
            engine_free(e);
            e = nullptr;
        }
        return rc;
    }
    e->groups.push_back(g);
    e->bound++;
    return OPTIM_OK;
}

void offload_unbind(optim_group* g) {
    if (!g->offload) return;
    OffloadBinding* b = g->offload;
    optim_offload* e = b->eng;
    if (b->slot >= 0) e->slots[b->slot].owner = nullptr;
    cudaFree(b->d_tables);
    delete b;
    g->offload = nullptr;
    if (e->library_owned) {
        std::lock_guard<std::mutex> lock(g_ring_mu);
        for (size_t i = 0; i < e->groups.size(); ++i)
            if (e->groups[i] == g) {
                e->groups.erase(e->groups.begin() + i);
                break;
            }
        if (--e->bound == 0) {
            // copies may still be queued on callers' copy streams: wait (bounded) for every
            // slot's last events as well as the ring's own streams before freeing the slots
            stream_wait_all(e);
            for (Slot& sl : e->slots)
                for (cudaEvent_t ev : {sl.h2d_done, sl.comp_done, sl.d2h_done}) wait_event(ev, kWaitTimeout, "staging slot");
            g_ring[e->device] = nullptr;
            engine_free(e);
        }
    } else {
        e->bound--;
    }
}

static int check_attachable(optim_group* g) {
    if (!offloadable(g->kind)) return set_error(OPTIM_EINVAL, "only NADAM, NADAM_F24, ADAN and ADAN_F24 groups can be offloaded");
    if (g->offload) return set_error(OPTIM_ESTATE, "group already attached");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    return OPTIM_OK;
}

static bool is_pinned_host(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

}  // namespace lmo

using namespace lmo;

extern "C" {

int optim_offload_create(size_t slot_bytes, int32_t n_slots, optim_offload_t** out) {
    if (!out || slot_bytes == 0 || n_slots < 2 || n_slots > 64)
        return set_error(OPTIM_EINVAL, "need out, slot_bytes > 0 and 2 <= n_slots <= 64");
    return engine_new(slot_bytes, n_slots, out);
}

int optim_offload_destroy(optim_offload_t* e) {
    if (!e) return set_error(OPTIM_EINVAL, "engine is NULL");
    if (e->library_owned) return set_error(OPTIM_EINVAL, "the library's own staging ring is freed with its last group");
    if (e->bound > 0) return set_error(OPTIM_ESTATE, "%d groups are still attached", e->bound);
    int rc = stream_wait_all(e);
    engine_free(e);
    return rc;
}

int optim_group_attach_offload(optim_group_t* g, optim_offload_t* e) {
    if (!g || !e) return set_error(OPTIM_EINVAL, "group or engine is NULL");
    int rc = check_attachable(g);
    if (rc) return rc;
    if (g->device != e->device) return set_error(OPTIM_EINVAL, "group and engine are on different devices");
    OffloadBinding* b = plan_binding(g);
    b->eng = e;
    for (int32_t i = 0; i < g->n; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        const size_t sz[3] = {b->sz_res[i], b->sz_m[i], b->sz_v[i]};
        const size_t off[3] = {b->off_res[i], b->off_m[i], b->off_v[i]};
        void* const ptr[3] = {d.res_u16, d.m, d.v};
        for (int k = 0; k < 3; ++k) {
            if (sz[k] == 0) continue;
            if (!is_pinned_host(ptr[k])) {
                delete b;
                return set_error(OPTIM_EINVAL, "tensor %d: offloaded states must be pinned host memory", i);
            }
            b->regions.push_back(Region{off[k], sz[k], static_cast<char*>(ptr[k])});
        }
    }
    if (b->need > e->slot_bytes) {
        const size_t need = b->need;
        delete b;
        return set_error(OPTIM_EINVAL, "group needs %zu staging bytes, slots hold %zu", need, e->slot_bytes);
    }
    rc = upload_tables(g, b);
    if (rc) {
        cudaFree(b->d_tables);
        delete b;
        return rc;
    }
    g->offload = b;
    e->bound++;
    return OPTIM_OK;
}

int optim_offload_layout(optim_group_t* g, int64_t* offsets, int64_t* total_bytes) {
    if (!g || !total_bytes) return set_error(OPTIM_EINVAL, "group or total_bytes is NULL");
    if (!offloadable(g->kind)) return set_error(OPTIM_EINVAL, "only NADAM, NADAM_F24, ADAN and ADAN_F24 groups can be offloaded");
    OffloadBinding* b = plan_binding(g);
    *total_bytes = (int64_t)b->need;
    if (offsets) {
        for (int32_t i = 0; i < g->n; ++i) {
            offsets[3 * i + 0] = b->sz_res[i] ? (int64_t)b->off_res[i] : -1;
            offsets[3 * i + 1] = b->sz_m[i] ? (int64_t)b->off_m[i] : -1;
            offsets[3 * i + 2] = b->sz_v[i] ? (int64_t)b->off_v[i] : -1;
        }
    }
    delete b;
    return OPTIM_OK;
}

int optim_group_attach_host(optim_group_t* g, void* image, size_t bytes) {
    if (!g || !image) return set_error(OPTIM_EINVAL, "group or image is NULL");
    int rc = check_attachable(g);
    if (!rc) rc = check_group_device(g);
    if (rc) return rc;
    if (!is_pinned_host(image)) return set_error(OPTIM_EINVAL, "the host image must be pinned host memory");
    OffloadBinding* b = plan_binding(g);
    if (bytes < b->need) {
        const size_t need = b->need;
        delete b;
        return set_error(OPTIM_EINVAL, "host image of %zu bytes, the group needs %zu", bytes, need);
    }
    b->image = true;
    b->regions.push_back(Region{0, b->need, static_cast<char*>(image)});
    // the states move into the image: earlier steps must be complete, then one copy per buffer
    rc = sync_group(g);
    for (int32_t i = 0; i < g->n && !rc; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        const size_t sz[3] = {b->sz_res[i], b->sz_m[i], b->sz_v[i]};
        const size_t off[3] = {b->off_res[i], b->off_m[i], b->off_v[i]};
        const void* const ptr[3] = {d.res_u16, d.m, d.v};
        for (int k = 0; k < 3 && !rc; ++k)
            if (sz[k]) rc = check_cuda(cudaMemcpy(static_cast<char*>(image) + off[k], ptr[k], sz[k], cudaMemcpyDefault),
                                       "state copy into the host image");
    }
    if (!rc) rc = ring_bind(g, b);
    if (rc) {
        cudaFree(b->d_tables);
        delete b;
        return rc;
    }
    g->offload = b;
    return OPTIM_OK;
}

int optim_offload_prefetch(optim_group_t* g, void* copy_stream) {
    if (!g || !g->offload) return set_error(OPTIM_EINVAL, "group is NULL or not offloaded");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    return prefetch(g, static_cast<cudaStream_t>(copy_stream));
}

int optim_offload_writeback(optim_group_t* g, void* copy_stream) {
    if (!g || !g->offload) return set_error(OPTIM_EINVAL, "group is NULL or not offloaded");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    OffloadBinding* b = g->offload;
    if (!b->image) return OPTIM_OK;           // engine-attached groups write back at each step's end
    if (b->slot < 0) return set_error(OPTIM_ESTATE, "the group's states are not on the device (prefetch first)");
    if (fault("d2h")) return set_error(OPTIM_ECUDA, "injected D2H copy failure");
    return writeback(g, static_cast<cudaStream_t>(copy_stream));
}

int optim_offload_sync(optim_offload_t* e, uint64_t* bytes_h2d, uint64_t* bytes_d2h) {
    if (!e) {
        int dev = 0;
        int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
        if (rc) return rc;
        std::lock_guard<std::mutex> lock(g_ring_mu);
        e = (dev >= 0 && dev < kMaxDevices) ? g_ring[dev] : nullptr;
        if (!e) {
            if (bytes_h2d) *bytes_h2d = 0;
            if (bytes_d2h) *bytes_d2h = 0;
            return OPTIM_OK;
        }
    }
    int rc = stream_wait_all(e);
    if (bytes_h2d) *bytes_h2d = e->bytes_h2d;
    if (bytes_d2h) *bytes_d2h = e->bytes_d2h;
    return rc;
}

}  // extern "C"
