// api.cu -- the C ABI of liblmopt.so: group handles, validation, per-step host scalars,
// gradient-pointer upload and kernel dispatch.  Declarations and contracts: include/lmopt.h.
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

#include "group.h"
#include "prodigy.h"

namespace lmo {

static thread_local char g_err[512] = "";

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int check_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return OPTIM_OK;
    return set_error(OPTIM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count() {
    static int cache[256] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

unsigned grid_for(int64_t units) {
    int64_t blocks = (units + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return (unsigned)(blocks < 1 ? 1 : blocks);
}

bool fault_injected(const char* what) {
    const char* f = std::getenv("LMOPT_FAULT_INJECT");
    return f && std::strcmp(f, what) == 0;
}

// Bounded host wait: polls the event until it completes or `timeout_s` passes.  With
// LMOPT_FAULT_INJECT=timeout every wait runs out at once (tests of the error path; nothing on
// the GPU is disturbed).
int wait_event(cudaEvent_t ev, double timeout_s, const char* what) {
    if (fault_injected("timeout")) return set_error(OPTIM_ETIMEOUT, "%s: no completion (injected timeout)", what);
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return OPTIM_OK;
        if (e != cudaErrorNotReady) return check_cuda(e, what);
        double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (dt > timeout_s) return set_error(OPTIM_ETIMEOUT, "%s: no completion after %.0f s", what, timeout_s);
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}


}  // namespace lmo

using namespace lmo;

static void group_free(optim_group* g) {
    if (!g) return;
    offload_unbind(g);
    prodigy_detach(g);
    for (int s = 0; s < 2; ++s) {
        if (g->stage_ev[s]) {
            cudaEventSynchronize(g->stage_ev[s]);
            cudaEventDestroy(g->stage_ev[s]);
        }
        if (g->h_stage[s]) cudaFreeHost(g->h_stage[s]);
    }
    if (g->sync_ev) cudaEventDestroy(g->sync_ev);
    cudaFree(g->d_tensors);
    cudaFree(g->d_grads);
    cudaFree(g->d_scales);
    cudaFree(g->d_chunks);
    cudaFree(g->d_nonfinite);
    cudaFree(g->d_zero_chunk);
    cudaFree(g->d_bar);
    factored_plan_free(g->fplan);
    delete g;
}

namespace lmo {
int check_group_device(const optim_group* g) {
    int dev = -1;
    int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev != g->device)
        return set_error(OPTIM_EINVAL, "group was created on device %d but device %d is current", g->device, dev);
    return OPTIM_OK;
}

// Bounded wait for the work of the group's last step call (on the stream it was enqueued on).
int sync_group(optim_group* g) {
    int rc = check_cuda(cudaEventRecord(g->sync_ev, g->last_stream), "sync event");
    if (rc) return rc;
    return wait_event(g->sync_ev, kWaitTimeout, "group stream");
}
}  // namespace lmo

static int validate_desc(const optim_tensor_desc_t& d, int32_t i, int32_t kind) {
    if (d.numel < 0) return set_error(OPTIM_EINVAL, "tensor %d: numel %lld < 0", i, (long long)d.numel);
    if (d.ndim < 1 || d.ndim > 4) return set_error(OPTIM_EINVAL, "tensor %d: ndim %d not in 1..4", i, d.ndim);
    int64_t prod = 1;
    for (int k = 0; k < d.ndim; ++k) {
        if (d.shape[k] < 0) return set_error(OPTIM_EINVAL, "tensor %d: negative dim", i);
        prod *= d.shape[k];
    }
    if (prod != d.numel)
        return set_error(OPTIM_EINVAL, "tensor %d: shape product %lld != numel %lld", i, (long long)prod,
                         (long long)d.numel);
    if (d.numel == 0) return OPTIM_OK;
    if (!d.w_bf16) return set_error(OPTIM_EINVAL, "tensor %d: w_bf16 is NULL", i);
    if (!is_aligned(d.w_bf16, 2) || (d.res_u16 && !is_aligned(d.res_u16, 2)))
        return set_error(OPTIM_EALIGN, "tensor %d: weight/residual not 2-byte aligned", i);
    if (kind == OPTIM_KIND_NADAM || kind == OPTIM_KIND_NADAM_F24) {
        if (!d.m || !d.v) return set_error(OPTIM_EINVAL, "tensor %d: m or v is NULL", i);
        size_t a = d.numel <= kSmall ? 4 : 2;
        if (!is_aligned(d.m, a) || !is_aligned(d.v, a))
            return set_error(OPTIM_EALIGN, "tensor %d: m/v not %zu-byte aligned", i, a);
    } else if (kind == OPTIM_KIND_ADAN || kind == OPTIM_KIND_ADAN_F24) {
        if (!d.m || !d.v) return set_error(OPTIM_EINVAL, "tensor %d: Adan state or previous gradient is NULL", i);
        if (!is_aligned(d.m, 4) || !is_aligned(d.v, 2))
            return set_error(OPTIM_EALIGN, "tensor %d: Adan buffers not aligned", i);
    } else {
        if (!d.v || (d.ndim >= 2 && !d.m)) return set_error(OPTIM_EINVAL, "tensor %d: factored state is NULL", i);
        if (!is_aligned(d.v, 4) || (d.m && !is_aligned(d.m, 4)))
            return set_error(OPTIM_EALIGN, "tensor %d: factored state not 4-byte aligned", i);
    }
    return OPTIM_OK;
}

template <class T>
static int dev_upload(T** dst, const std::vector<T>& src, const char* what) {
    size_t bytes = src.size() * sizeof(T);
    if (bytes == 0) bytes = sizeof(T);
    if (cudaMalloc(reinterpret_cast<void**>(dst), bytes) != cudaSuccess) {
        cudaGetLastError();
        return set_error(OPTIM_ENOMEM, "cudaMalloc(%zu) for %s failed", bytes, what);
    }
    if (src.empty()) return check_cuda(cudaMemset(*dst, 0, bytes), what);
    return check_cuda(cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice), what);
}

static int upload_grads(optim_group* g, const void* const* grads, cudaStream_t s) {
    if (g->grads_valid && std::memcmp(g->cur_grads.data(), grads, sizeof(void*) * g->n) == 0)
        return OPTIM_OK;
    const int slot = g->stage_slot;
    int rc = wait_event(g->stage_ev[slot], kWaitTimeout, "gradient table staging slot");
    if (rc) return rc;
    std::memcpy(g->h_stage[slot], grads, sizeof(void*) * g->n);
    rc = check_cuda(cudaMemcpyAsync(g->d_grads, g->h_stage[slot], sizeof(void*) * g->n,
                                    cudaMemcpyHostToDevice, s), "gradient table upload");
    if (rc) return rc;
    rc = check_cuda(cudaEventRecord(g->stage_ev[slot], s), "gradient table event");
    if (rc) return rc;
    g->stage_slot ^= 1;
    std::memcpy(g->cur_grads.data(), grads, sizeof(void*) * g->n);
    g->grads_valid = true;
    return OPTIM_OK;
}

static int validate_grads(const optim_group* g, const void* const* grads) {
    if (!grads) return set_error(OPTIM_EINVAL, "grads_bf16 is NULL");
    for (int32_t i = 0; i < g->n; ++i) {
        if (g->desc[i].numel == 0) continue;
        if (!grads[i]) return set_error(OPTIM_EINVAL, "gradient %d is NULL", i);
        if (!is_aligned(grads[i], 2)) return set_error(OPTIM_EALIGN, "gradient %d not 2-byte aligned", i);
    }
    return OPTIM_OK;
}

static bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.0f; }

// What the update kernels take for granted about a group's chunk table, checked once when it is
// built: every entry names a tensor of the group, the u16-state (large) tensors' chunks come
// first, and each tensor's chunks are 0, 1, ..., ceil(numel / chunk) - 1 in that order, so that
// every chunk starts inside its tensor and every element lies in exactly one chunk.
static int check_chunk_table(const optim_tensor_desc_t* t, int32_t n, const std::vector<Chunk>& chunks,
                             int64_t chunk, int32_t n_large) {
    std::vector<int64_t> next(n, 0);
    for (size_t j = 0; j < chunks.size(); ++j) {
        const Chunk c = chunks[j];
        if (c.tensor < 0 || c.tensor >= n)
            return set_error(OPTIM_EINVAL, "internal: chunk table entry %zu names tensor %d of %d", j, c.tensor, n);
        const int64_t ne = t[c.tensor].numel;
        if (((int64_t)j < n_large) != (ne > kSmall))
            return set_error(OPTIM_EINVAL, "internal: chunk table entry %zu outside its tensor's section", j);
        if (c.index != next[c.tensor] || (int64_t)c.index * chunk >= ne)
            return set_error(OPTIM_EINVAL, "internal: chunk table entry %zu (tensor %d, chunk %d) out of order or "
                             "past the tensor's end", j, c.tensor, c.index);
        ++next[c.tensor];
    }
    for (int32_t i = 0; i < n; ++i)
        if (next[i] != (t[i].numel + chunk - 1) / chunk)
            return set_error(OPTIM_EINVAL, "internal: tensor %d covered by %lld chunks", i, (long long)next[i]);
    return OPTIM_OK;
}

extern "C" {

const char* optim_last_error(void) { return g_err; }

int optim_group_create(const optim_tensor_desc_t* tensors, int32_t n, int32_t kind, optim_group_t** out) {
    if (!out) return set_error(OPTIM_EINVAL, "out is NULL");
    *out = nullptr;
    if (!tensors || n < 1) return set_error(OPTIM_EINVAL, "need n >= 1 tensors");
    if (kind != OPTIM_KIND_NADAM && kind != OPTIM_KIND_FACTORED && kind != OPTIM_KIND_NADAM_F24 &&
        kind != OPTIM_KIND_ADAN && kind != OPTIM_KIND_ADAN_F24)
        return set_error(OPTIM_EINVAL, "unknown group kind %d", kind);
    for (int32_t i = 0; i < n; ++i) {
        int rc = validate_desc(tensors[i], i, kind);
        if (rc) return rc;
    }
    optim_group* g = new optim_group();
    g->kind = kind;
    g->n = n;
    g->desc.assign(tensors, tensors + n);
    g->cur_grads.assign(n, nullptr);
    int rc = check_cuda(cudaGetDevice(&g->device), "cudaGetDevice");
    if (!rc) {
        std::vector<TensorRec> recs(n);
        std::vector<Chunk> chunks;
        for (int32_t i = 0; i < n; ++i) {
            const optim_tensor_desc_t& d = tensors[i];
            TensorRec& r = recs[i];
            r.w = static_cast<uint16_t*>(d.w_bf16);
            r.res = static_cast<uint16_t*>(d.res_u16);
            r.m = d.m;
            r.v = d.v;
            r.numel = d.numel;
            r.flags = (d.numel <= kSmall ? kFlagSmall : 0) | (d.res_u16 ? kFlagRes : 0);
            r.pad = 0;
        }
        if (kind != OPTIM_KIND_FACTORED) {
            // chunks of kChunkU16 elements for NAdam u16 groups, kChunk for f24 and Adan groups;
            // a group whose chunks would not give every SM a CTA (two for the
            // kinds without the one-launch step) is cut finer, down to kChunkMin: the small case
            // then spreads over the whole GPU (for the one-launch step one CTA per SM measured
            // faster than two: fewer, longer CTAs share the per-CTA prologue and the instruction
            // fetch of the short launch)
            auto count = [&](int64_t ch) {
                int64_t c = 0;
                for (int32_t i = 0; i < n; ++i) c += (tensors[i].numel + ch - 1) / ch;
                return c;
            };
            const int64_t per_sm = kind == OPTIM_KIND_NADAM ? 1 : 2;
            g->chunk = kind == OPTIM_KIND_NADAM ? kChunkU16 : kChunk;
            while (g->chunk > kChunkMin && count(g->chunk) < per_sm * (int64_t)sm_count()) g->chunk /= 2;
            for (int pass = 0; pass < 2; ++pass) {   // u16-state tensors first, then fp32-state
                for (int32_t i = 0; i < n; ++i) {
                    const int64_t ne = tensors[i].numel;
                    if (ne == 0 || (pass == 0) != (ne > kSmall)) continue;
                    const int64_t nc = (ne + g->chunk - 1) / g->chunk;
                    for (int64_t c = 0; c < nc; ++c) chunks.push_back(Chunk{i, (int32_t)c});
                }
                if (pass == 0) g->n_chunks_large = (int32_t)chunks.size();
            }
            if (chunks.size() > (size_t)INT32_MAX) rc = set_error(OPTIM_EINVAL, "group too large");
            g->n_chunks_total = (int32_t)chunks.size();
            if (!rc) rc = check_chunk_table(tensors, n, chunks, g->chunk, g->n_chunks_large);
        }
        if (!rc) rc = dev_upload(&g->d_tensors, recs, "tensor table");
        if (!rc) rc = dev_upload(&g->d_chunks, chunks, "chunk table");
        if (!rc) rc = dev_upload(&g->d_scales, std::vector<ScaleRec>(n, ScaleRec{}), "scale table");
        if (!rc) rc = dev_upload(&g->d_nonfinite, std::vector<unsigned long long>(1, 0ull), "counter");
        if (!rc) rc = dev_upload(&g->d_zero_chunk, std::vector<uint8_t>(std::max<int32_t>(g->n_chunks_large, 1), 1), "zero flags");
        if (!rc) rc = dev_upload(&g->d_grads, std::vector<const uint16_t*>(n, nullptr), "gradient table");
        if (!rc && kind == OPTIM_KIND_NADAM) rc = dev_upload(&g->d_bar, std::vector<unsigned>(1, 0u), "barrier counter");
        for (int s = 0; s < 2 && !rc; ++s) {
            if (cudaHostAlloc(reinterpret_cast<void**>(&g->h_stage[s]), sizeof(void*) * n, cudaHostAllocDefault) != cudaSuccess) {
                cudaGetLastError();
                rc = set_error(OPTIM_ENOMEM, "pinned staging allocation failed");
                break;
            }
            rc = check_cuda(cudaEventCreateWithFlags(&g->stage_ev[s], cudaEventDisableTiming), "event");
        }
        if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&g->sync_ev, cudaEventDisableTiming), "event");
        if (!rc && kind == OPTIM_KIND_FACTORED) rc = factored_plan_build(g->fplan, g->desc);
    }
    if (rc) {
        group_free(g);
        return rc;
    }
    *out = g;
    if (const char* vb = std::getenv("LMOPT_VERBOSE"); vb && std::strcmp(vb, "1") == 0) {
        // one line per group: what was switched on (the Kahan residual, the moment storage)
        int64_t numel = 0, res = 0;
        for (int32_t i = 0; i < n; ++i) {
            numel += tensors[i].numel;
            res += tensors[i].res_u16 != nullptr && tensors[i].numel > 0;
        }
        static const char* const names[] = {"nadam u16", "factored", "nadam f24", "adan fp32", "adan f24"};
        std::fprintf(stderr, "lmopt: group of %d tensors, %lld elements, %s states, Kahan residual on %lld "
                     "tensors, device %d", n, (long long)numel, names[kind], (long long)res, g->device);
        if (kind != OPTIM_KIND_FACTORED)
            std::fprintf(stderr, ", %d chunks of %lld elements (%d u16-state)", g->n_chunks_total,
                         (long long)g->chunk, g->n_chunks_large);
        std::fprintf(stderr, "\n");
    }
    return OPTIM_OK;
}

int optim_group_destroy(optim_group_t* g) {
    if (!g) return set_error(OPTIM_EINVAL, "group is NULL");
    group_free(g);
    return OPTIM_OK;
}

}  // extern "C"

// Validation, per-step scalars, gradient upload and (unless `fused`) the pre-pass of a NAdam
// step; with `fused` the pre-pass is left to the one-launch step enqueued by nadam_end.
static int nadam_begin(optim_group_t* g, const void* const* grads, int64_t step, const optim_nadam_hparams_t* hp,
                       void* stream, float* exchange, bool fused) {
    if (!g || !hp) return set_error(OPTIM_EINVAL, "group or hparams is NULL");
    if (g->kind != OPTIM_KIND_NADAM && g->kind != OPTIM_KIND_NADAM_F24)
        return set_error(OPTIM_EINVAL, "not a NADAM group");
    if (g->pending) return set_error(OPTIM_ESTATE, "step %lld was begun and not ended", (long long)g->pending_step);
    if (step != g->last_step + 1)
        return set_error(OPTIM_EINVAL, "step %lld but the group expects %lld", (long long)step,
                         (long long)(g->last_step + 1));
    if (!finite_nonneg(hp->lr) || !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) ||
        !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) || !finite_nonneg(hp->eps) ||
        !finite_nonneg(hp->weight_decay) || !finite_nonneg(hp->momentum_decay) ||
        (hp->wd_mode != 0 && hp->wd_mode != 1) || (hp->nesterov != 0 && hp->nesterov != 1) ||
        (hp->stochastic_rounding != 0 && hp->stochastic_rounding != 1))
        return set_error(OPTIM_EINVAL, "invalid NAdam hyper-parameters (wd_mode must be 0 or 1)");
    if (exchange && !is_aligned(exchange, 4)) return set_error(OPTIM_EALIGN, "exchange buffer not 4-byte aligned");
    int rc = check_group_device(g);
    if (!rc) rc = validate_grads(g, grads);
    if (rc) return rc;

    // per-step scalars: double precision, one rounding to fp32 each
    const double b1 = hp->beta1, b2 = hp->beta2, td = (double)step;
    double mu_product = g->mu_product;
    NadamScalars k{};
    k.lr = hp->lr;
    k.b1 = hp->beta1;
    k.omb1 = (float)(1.0 - b1);
    k.b2 = hp->beta2;
    k.omb2 = (float)(1.0 - b2);
    k.eps = hp->eps;
    k.lr_wd = (float)((double)hp->lr * (double)hp->weight_decay);
    k.decoupled = hp->wd_mode == 1;
    k.k2 = (float)(1.0 / std::sqrt(1.0 - std::pow(b2, td)));
    if (hp->nesterov) {
        const double psi = hp->momentum_decay;
        const double mu = b1 * (1.0 - 0.5 * std::pow(0.96, td * psi));
        const double mu_next = b1 * (1.0 - 0.5 * std::pow(0.96, (td + 1.0) * psi));
        mu_product = mu_product * mu;
        k.c_g = (float)((1.0 - mu) / (1.0 - mu_product));
        k.c_m = (float)(mu_next / (1.0 - mu_product * mu_next));
    } else {
        k.c_m = (float)(1.0 / (1.0 - std::pow(b1, td)));
        k.c_g = 0.0f;
    }
    k.parity = g->next_parity;
    k.sr = hp->stochastic_rounding;
    k.seed = hp->seed;
    k.step = (uint64_t)step;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = upload_grads(g, grads, s);
    if (rc) return rc;
    const TensorRec* table = g->d_tensors;
    if (g->offload) {
        rc = offload_step_begin(g, s, &table);
        if (rc) return rc;
    }
    NadamLaunch L{table, g->d_grads, g->d_scales, g->d_chunks, g->d_nonfinite,
                  g->n_chunks_large, g->n_chunks_total, g->kind == OPTIM_KIND_NADAM_F24, g->d_zero_chunk, g->chunk};
    if (!fused) rc = launch_nadam_prepass(L, k, s);
    if (!rc && exchange) rc = launch_scales_gather(g->d_scales, exchange, g->n, k.parity, s);
    if (rc) return rc;
    g->pending = true;
    g->pending_fused = fused;
    g->pending_step = step;
    g->pending_mu = mu_product;
    g->pending_k = k;
    g->pending_table = table;
    g->pending_stream = s;
    return OPTIM_OK;
}

extern "C" {

int optim_step_nadam_begin(optim_group_t* g, const void* const* grads, int64_t step,
                           const optim_nadam_hparams_t* hp, void* stream, float* exchange) {
    return nadam_begin(g, grads, step, hp, stream, exchange, false);
}

int optim_step_nadam_end(optim_group_t* g, const float* exchange, void* stream) {
    if (!g) return set_error(OPTIM_EINVAL, "group is NULL");
    if (!g->pending) return set_error(OPTIM_ESTATE, "no NAdam step was begun on this group");
    if (exchange && !is_aligned(exchange, 4)) return set_error(OPTIM_EALIGN, "exchange buffer not 4-byte aligned");
    int rc = check_group_device(g);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const NadamScalars& k = g->pending_k;
    NadamLaunch L{g->pending_table, g->d_grads, g->d_scales, g->d_chunks, g->d_nonfinite,
                  g->n_chunks_large, g->n_chunks_total, g->kind == OPTIM_KIND_NADAM_F24, g->d_zero_chunk, g->chunk};
    if (exchange) rc = launch_scales_scatter(g->d_scales, exchange, g->n, k.parity, s);
    if (!rc && g->pending_fused) {
        if (g->profile_ev) rc = check_cuda(cudaEventRecord(g->profile_ev, s), "profile event");
        const unsigned target = g->bar_total + (unsigned)g->n_chunks_total;
        if (!rc) rc = launch_nadam_fused(L, k, s, g->d_bar, target);
        if (!rc) g->bar_total = target;
    } else if (!rc) {
        rc = launch_nadam_update(L, k, s, g->profile_ev);
    }
    if (rc) return rc;
    g->pending = false;
    g->pending_fused = false;
    g->last_step = g->pending_step;
    g->mu_product = g->pending_mu;
    g->next_parity ^= 1;
    g->last_stream = s;
    if (g->offload) return offload_step_end(g, s);
    return OPTIM_OK;
}

// One launch when the group's chunks all fit on the GPU at once (u16 groups with a pre-pass).
static bool nadam_fusable(const optim_group* g, const optim_nadam_hparams_t* hp) {
    if (!g || !hp || g->kind != OPTIM_KIND_NADAM || !g->d_bar || g->n_chunks_large == 0) return false;
    const int cap = nadam_fused_capacity(hp->stochastic_rounding == 1);
    return g->n_chunks_total <= cap;
}

int optim_step_nadam_kahan(optim_group_t* g, const void* const* grads, int64_t step,
                           const optim_nadam_hparams_t* hp, void* stream) {
    int rc = nadam_begin(g, grads, step, hp, stream, nullptr, nadam_fusable(g, hp));
    if (rc) return rc;
    return optim_step_nadam_end(g, nullptr, stream);
}

int optim_query_launches(optim_group_t* g, const optim_nadam_hparams_t* hp, int32_t* launches) {
    if (!g || !launches) return set_error(OPTIM_EINVAL, "group or output is NULL");
    if (g->kind == OPTIM_KIND_NADAM) {
        if (!hp) return set_error(OPTIM_EINVAL, "hparams is NULL");
        *launches = nadam_fusable(g, hp) ? 1 : (g->n_chunks_large > 0 ? 2 : 1);
    } else if (g->kind == OPTIM_KIND_FACTORED) {
        return set_error(OPTIM_EINVAL, "factored groups launch per wave (see optim_step_factored)");
    } else {
        *launches = 1;
    }
    return OPTIM_OK;
}

int optim_step_adan(optim_group_t* g, const void* const* grads, int64_t step, const optim_adan_hparams_t* hp,
                    void* stream) {
    if (!g || !hp) return set_error(OPTIM_EINVAL, "group or hparams is NULL");
    if (g->kind != OPTIM_KIND_ADAN && g->kind != OPTIM_KIND_ADAN_F24) return set_error(OPTIM_EINVAL, "not an ADAN group");
    if (step != g->last_step + 1)
        return set_error(OPTIM_EINVAL, "step %lld but the group expects %lld", (long long)step,
                         (long long)(g->last_step + 1));
    auto unit = [](float x) { return x >= 0.0f && x <= 1.0f; };
    if (!finite_nonneg(hp->lr) || !unit(hp->beta1) || !unit(hp->beta2) || !unit(hp->beta3) ||
        !finite_nonneg(hp->eps) || !finite_nonneg(hp->weight_decay) ||
        (hp->stochastic_rounding != 0 && hp->stochastic_rounding != 1))
        return set_error(OPTIM_EINVAL, "invalid Adan hyper-parameters");
    int rc = check_group_device(g);
    if (!rc) rc = validate_grads(g, grads);
    if (rc) return rc;
    AdanScalars k{};
    k.lr = hp->lr;
    k.b1 = hp->beta1;
    k.omb1 = (float)(1.0 - (double)hp->beta1);
    k.b2 = hp->beta2;
    k.omb2 = (float)(1.0 - (double)hp->beta2);
    k.b3 = hp->beta3;
    k.omb3 = (float)(1.0 - (double)hp->beta3);
    k.eps = hp->eps;
    k.inv_decay = (float)(1.0 / (1.0 + (double)hp->lr * (double)hp->weight_decay));
    k.sr = hp->stochastic_rounding;
    k.step = step;
    k.seed = hp->seed;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = upload_grads(g, grads, s);
    if (rc) return rc;
    const TensorRec* table = g->d_tensors;
    if (g->offload) {
        rc = offload_step_begin(g, s, &table);
        if (rc) return rc;
    }
    NadamLaunch L{table, g->d_grads, g->d_scales, g->d_chunks, g->d_nonfinite, g->n_chunks_large,
                  g->n_chunks_total, g->kind == OPTIM_KIND_ADAN_F24, nullptr, g->chunk};
    rc = launch_adan_step(L, k, s);
    if (rc) return rc;
    g->last_step = step;
    g->last_stream = s;
    if (g->offload) return offload_step_end(g, s);
    return OPTIM_OK;
}

int optim_step_factored(optim_group_t* g, const void* const* grads, int64_t step,
                        const optim_factored_hparams_t* hp, void* stream) {
    if (!g || !hp) return set_error(OPTIM_EINVAL, "group or hparams is NULL");
    if (g->kind != OPTIM_KIND_FACTORED) return set_error(OPTIM_EINVAL, "not a FACTORED group");
    if (step != g->last_step + 1)
        return set_error(OPTIM_EINVAL, "step %lld but the group expects %lld", (long long)step,
                         (long long)(g->last_step + 1));
    if (!finite_nonneg(hp->lr) || !(hp->clip_threshold > 0.0f) || !std::isfinite(hp->clip_threshold) ||
        !finite_nonneg(hp->weight_decay) || !finite_nonneg(hp->eps1) || !finite_nonneg(hp->eps2) ||
        (hp->mode != 0 && hp->mode != 1) || !std::isfinite(hp->decay_rate) ||
        (hp->mode == 1 && (!(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) || (!g->prodigy && !finite_nonneg(hp->d)))))
        return set_error(OPTIM_EINVAL, "invalid factored hyper-parameters");
    if (g->prodigy && hp->mode != 1)
        return set_error(OPTIM_EINVAL, "a group attached to a Prodigy controller steps in mode 1");
    int rc = check_group_device(g);
    if (!rc) rc = validate_grads(g, grads);
    if (rc) return rc;

    FactoredScalars k = factored_scalars(hp, step, g->prodigy ? 1.0f : hp->d);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = upload_grads(g, grads, s);
    if (rc) return rc;
    cudaEvent_t apply_wait = nullptr;
    if (g->prodigy) {
        rc = prodigy_step_begin(g, hp, s, &k.kdev, &apply_wait);
        if (rc) {
            prodigy_step_join(g, s);
            return rc;
        }
    }
    rc = launch_factored_step(g->fplan, g->d_grads, k, s, g->profile_ev, g->d_nonfinite, apply_wait);
    if (g->prodigy) {
        const int r2 = prodigy_step_join(g, s);
        if (!rc) rc = r2;
    }
    if (rc) return rc;
    g->last_step = step;
    g->last_stream = s;
    return OPTIM_OK;
}


int optim_query_scales(optim_group_t* g, float* host_out) {
    if (!g || !host_out) return set_error(OPTIM_EINVAL, "group or output is NULL");
    if (g->kind != OPTIM_KIND_NADAM) return set_error(OPTIM_EINVAL, "not a NADAM group");
    int rc = check_group_device(g);
    if (!rc) rc = sync_group(g);
    if (rc) return rc;
    std::vector<ScaleRec> recs(g->n);
    rc = check_cuda(cudaMemcpy(recs.data(), g->d_scales, sizeof(ScaleRec) * g->n, cudaMemcpyDeviceToHost),
                    "scale download");
    if (rc) return rc;
    const int lp = g->next_parity ^ 1;
    for (int32_t i = 0; i < g->n; ++i) {
        float am, av;
        std::memcpy(&am, &recs[i].a_m[lp], 4);
        std::memcpy(&av, &recs[i].a_v[lp], 4);
        host_out[4 * i + 0] = recs[i].s_m[lp];
        host_out[4 * i + 1] = recs[i].s_v[lp];
        host_out[4 * i + 2] = am;
        host_out[4 * i + 3] = av;
    }
    return OPTIM_OK;
}

int optim_set_scales(optim_group_t* g, const float* host_in) {
    if (!g || !host_in) return set_error(OPTIM_EINVAL, "group or input is NULL");
    if (g->kind != OPTIM_KIND_NADAM) return set_error(OPTIM_EINVAL, "not a NADAM group");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    int rc = check_group_device(g);
    if (!rc) rc = sync_group(g);
    if (rc) return rc;
    std::vector<ScaleRec> recs(g->n, ScaleRec{});
    const int lp = g->next_parity ^ 1;
    for (int32_t i = 0; i < g->n; ++i) {
        for (int k = 0; k < 4; ++k)
            if (!(host_in[4 * i + k] >= 0.0f) || !std::isfinite(host_in[4 * i + k]))
                return set_error(OPTIM_EINVAL, "scale record %d is negative or not finite", i);
        recs[i].s_m[lp] = host_in[4 * i + 0];
        recs[i].s_v[lp] = host_in[4 * i + 1];
        std::memcpy(&recs[i].a_m[lp], &host_in[4 * i + 2], 4);
        std::memcpy(&recs[i].a_v[lp], &host_in[4 * i + 3], 4);
    }
    return check_cuda(cudaMemcpy(g->d_scales, recs.data(), sizeof(ScaleRec) * g->n, cudaMemcpyHostToDevice),
                      "scale upload");
}

int optim_group_get_step(optim_group_t* g, int64_t* step, double* mu_product) {
    if (!g || !step || !mu_product) return set_error(OPTIM_EINVAL, "NULL argument");
    *step = g->last_step;
    *mu_product = g->mu_product;
    return OPTIM_OK;
}

int optim_group_set_step(optim_group_t* g, int64_t step, double mu_product) {
    if (!g || step < 0 || !std::isfinite(mu_product)) return set_error(OPTIM_EINVAL, "bad step or mu product");
    if (g->pending) return set_error(OPTIM_ESTATE, "a NAdam step was begun and not ended");
    g->last_step = step;
    g->mu_product = mu_product;
    return OPTIM_OK;
}

int optim_group_set_profile_event(optim_group_t* g, void* event) {
    if (!g) return set_error(OPTIM_EINVAL, "group is NULL");
    g->profile_ev = static_cast<cudaEvent_t>(event);
    return OPTIM_OK;
}

int optim_query_nonfinite(optim_group_t* g, uint64_t* count) {
    if (!g || !count) return set_error(OPTIM_EINVAL, "NULL argument");
    int rc = check_group_device(g);
    if (!rc) rc = sync_group(g);
    if (rc) return rc;
    unsigned long long c = 0;
    rc = check_cuda(cudaMemcpy(&c, g->d_nonfinite, sizeof c, cudaMemcpyDeviceToHost), "counter download");
    *count = c;
    return rc;
}

// ---------------------------------------------------------------- stand-alone codec entry points
static int check_buf(const void* p, size_t align, const char* name) {
    if (!p) return set_error(OPTIM_EINVAL, "%s is NULL", name);
    if (!is_aligned(p, align)) return set_error(OPTIM_EALIGN, "%s not %zu-byte aligned", name, align);
    return OPTIM_OK;
}

int state_pack_u16(const float* src, uint16_t* codes, float* scale, int64_t n, int32_t is_signed, void* stream) {
    if (n < 0 || (is_signed != 0 && is_signed != 1)) return set_error(OPTIM_EINVAL, "bad n or is_signed");
    int rc = check_buf(scale, 4, "scale");
    if (rc) return rc;
    if (n > 0 && ((rc = check_buf(src, 4, "src")) || (rc = check_buf(codes, 2, "codes")))) return rc;
    return launch_state_pack(src, codes, scale, n, is_signed, static_cast<cudaStream_t>(stream));
}

int state_unpack_u16(const uint16_t* codes, const float* scale, float* dst, int64_t n, int32_t is_signed,
                     void* stream) {
    if (n < 0 || (is_signed != 0 && is_signed != 1)) return set_error(OPTIM_EINVAL, "bad n or is_signed");
    if (n == 0) return OPTIM_OK;
    int rc;
    if ((rc = check_buf(codes, 2, "codes")) || (rc = check_buf(scale, 4, "scale")) || (rc = check_buf(dst, 4, "dst")))
        return rc;
    return launch_state_unpack(codes, scale, dst, n, is_signed, static_cast<cudaStream_t>(stream));
}

int optim_kahan_split(const float* src, uint16_t* hi, uint16_t* lo, int64_t n, void* stream) {
    if (n < 0) return set_error(OPTIM_EINVAL, "n < 0");
    if (n == 0) return OPTIM_OK;
    int rc;
    if ((rc = check_buf(src, 4, "src")) || (rc = check_buf(hi, 2, "hi")) || (rc = check_buf(lo, 2, "lo"))) return rc;
    return launch_kahan_split(src, hi, lo, n, static_cast<cudaStream_t>(stream));
}

int optim_kahan_merge(const uint16_t* hi, const uint16_t* lo, float* dst, int64_t n, void* stream) {
    if (n < 0) return set_error(OPTIM_EINVAL, "n < 0");
    if (n == 0) return OPTIM_OK;
    int rc;
    if ((rc = check_buf(hi, 2, "hi")) || (rc = check_buf(lo, 2, "lo")) || (rc = check_buf(dst, 4, "dst"))) return rc;
    return launch_kahan_merge(hi, lo, dst, n, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
