// prodigy.cu -- Prodigy's step-size estimate d over FACTORED groups (mode 1).
//
// The pages discuss Prodigy's d (prodigy PR #25, "more VRAM savings: no first moment and
// factored second moment": d0, the numerator built from p - p0, "s, which is the denominator in
// the calculation of d_hat", EMAs scaled by d; the slicing of PR #22) without printing its
// update.  This follows the Adam form of Prodigy (Mishchenko, Defazio, "Prodigy: An
// Expeditiously Adaptive Parameter-Free Learner", 2023) with beta1 = 0.  Per step k with d_k, for
// every sampled element e of every attached tensor, before the tensor's update:
//     dot += g_e (p0_e - x_e),     s_e = beta3 s_e + fl(lr d_k^2) g_e,     l1 += |s_e|
// and at the end of the step, over all attached groups:
//     r = beta3 r + sum_groups (lr d_k^2) dot,     d_{k+1} = max(d_k, r / l1)  (if l1 > 0).
// Sampled elements: the 64-element blocks of a tensor's flat elements whose block index is a
// multiple of slice_p; p0 and s hold them in order, 64 per sampled block.
//
// Work per step, per group call: a one-thread kernel writing the group's d-dependent scalars (read
// by the factored kernels after their programmatic-launch wait), and the statistics kernel on
// the group's own stream, concurrent with the factored kernels until their update kernels, which
// wait for it (it reads the weights they overwrite); per controller step, a one-CTA reduction.  The statistics
// touch 1/slice_p of the weights and gradients (whole 128-byte lines: 64 bf16 per block) and
// read/write p0 and s (12 bytes per sampled element).  Sums: fp32 over a thread's 32 entries of
// an item, compensated fp32 over its items, double across threads, CTAs and groups, each in a
// fixed order (the grid is fixed when the group attaches).
#include <algorithm>
#include <cmath>
#include <vector>

#include "group.h"
#include "prodigy.h"

namespace lmo {
namespace {

constexpr int kPdThreads = 256;
constexpr int kPdPerThread = 32;
constexpr int64_t kPdPerCta = (int64_t)kPdThreads * kPdPerThread;   // sampled entries per CTA
constexpr int kPdEndThreads = 1024;
// Statistics CTAs per SM (persistent grid).  A sparse sample (slice_p >= 4) is a small share of
// the step and runs beside the factored kernels up to their update, so it takes one CTA per SM
// and leaves them room (sdxl_like, slice_p 11: 6.87 ms per step against 6.98 with four); a dense
// one is as large as the step itself and takes four (slice_p 1: 13.0 against 14.7 ms with one).
constexpr int kPdCtasPerSmSparse = 1;
constexpr int kPdCtasPerSmDense = 4;

struct PdTensor {
    const uint16_t* w;
    const uint16_t* res;
    float* p0;
    float* s;
    int64_t numel;
    int64_t len;       // sampled entries (a multiple of 64)
};

struct PdItem {
    int32_t tensor;
    int32_t chunk;     // entries [chunk * kPdPerCta, ...) of the tensor
};

struct PdState {
    double d, r;
};

struct PdStep {
    float lr, beta2, wd, beta3;
    int32_t slice_p;
    int32_t n_items;
};

__device__ __forceinline__ int64_t sampled_element(int64_t j, int32_t slice_p) {
    return (j >> 6) * (int64_t)slice_p * 64 + (j & 63);
}

__device__ __forceinline__ float master(const PdTensor& t, int64_t e) {
    const uint32_t hi = t.w[e];
    return t.res ? __uint_as_float((hi << 16) | t.res[e]) : bf16_to_f32(hi);
}

// Block-wide double sum in a fixed tree; result valid in thread 0.
template <int kN>
__device__ double block_sum_f64(double x, double* sm /* kN / 32 */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    double y = 0.0;
    if (warp == 0) {
        y = lane < kN / 32 ? sm[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
    }
    __syncthreads();
    return y;
}

__global__ void __launch_bounds__(kPdThreads) k_pd_snapshot(const PdTensor* T, const PdItem* items, int32_t slice_p) {
    const PdItem it = items[blockIdx.x];
    const PdTensor t = T[it.tensor];
    const int64_t j0 = (int64_t)it.chunk * kPdPerCta;
    const int64_t j1 = t.len < j0 + kPdPerCta ? t.len : j0 + kPdPerCta;
    for (int64_t j = j0 + threadIdx.x; j < j1; j += kPdThreads) {
        const int64_t e = sampled_element(j, slice_p);
        t.p0[j] = e < t.numel ? master(t, e) : 0.0f;
        t.s[j] = 0.0f;
    }
}

// The statistics of one sampled entry (element e of the tensor, entry j of p0 / s).
__device__ __forceinline__ void pd_entry(float x, float gg, float p0, float& s, float beta3, float cs, float& dot,
                                         float& l1) {
    dot = __fadd_rn(dot, __fmul_rn(gg, __fsub_rn(p0, x)));
    s = __fadd_rn(__fmul_rn(beta3, s), __fmul_rn(cs, gg));
    l1 = __fadd_rn(l1, fabsf(s));
}

// One thread: the group's d-dependent scalars of the step, the same values as the host scalars
// of a mode-1 step with d = fl32(d).
__global__ void k_pd_scalars(const PdState* st, PdStep p, FactoredDevScalars* kdev) {
    const float df = (float)st->d;
    FactoredDevScalars v;
    v.alpha = (float)((double)df * (double)df * (1.0 - (double)p.beta2));
    v.lr_eff = (float)((double)df * (double)p.lr);
    v.nwdlr = (float)(-(double)p.wd * (double)v.lr_eff);
    v.unum = df;
    *kdev = v;
}

// Neumaier-compensated fp32 accumulation (a thread's sum over its items).
struct PdComp {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float t = __fadd_rn(s, x);
        if (fabsf(s) >= fabsf(x)) c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), x));
        else c = __fadd_rn(c, __fadd_rn(__fsub_rn(x, t), s));
        s = t;
    }
    __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

struct Pd8 {
    uint4 W, R, G;
    float4 P0, P1, S0, S1;
};
__device__ __forceinline__ void pd_load8(const PdTensor& t, const uint16_t* __restrict__ g, int64_t j, int64_t e, Pd8& v) {
    v.W = ld_stream(reinterpret_cast<const uint4*>(t.w + e));
    v.R = t.res ? ld_stream(reinterpret_cast<const uint4*>(t.res + e)) : make_uint4(0, 0, 0, 0);
    v.G = __ldcg(reinterpret_cast<const uint4*>(g + e));
    v.P0 = ld_stream(reinterpret_cast<const float4*>(t.p0 + j));
    v.P1 = ld_stream(reinterpret_cast<const float4*>(t.p0 + j + 4));
    v.S0 = ld_stream(reinterpret_cast<const float4*>(t.s + j));
    v.S1 = ld_stream(reinterpret_cast<const float4*>(t.s + j + 4));
}
__device__ __forceinline__ void pd_comp8(const PdTensor& t, int64_t j, const Pd8& v, float beta3, float cs, float& dot,
                                         float& l1) {
    const bool has_res = t.res != nullptr;
    const uint32_t w32[4] = {v.W.x, v.W.y, v.W.z, v.W.w}, r32[4] = {v.R.x, v.R.y, v.R.z, v.R.w};
    const uint32_t g32[4] = {v.G.x, v.G.y, v.G.z, v.G.w};
    const float pv[8] = {v.P0.x, v.P0.y, v.P0.z, v.P0.w, v.P1.x, v.P1.y, v.P1.z, v.P1.w};
    float sv[8] = {v.S0.x, v.S0.y, v.S0.z, v.S0.w, v.S1.x, v.S1.y, v.S1.z, v.S1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int sh = 16 * (q & 1);
        const uint32_t hw = (w32[q >> 1] >> sh) & 0xFFFFu, lw = (r32[q >> 1] >> sh) & 0xFFFFu;
        const float x = has_res ? __uint_as_float((hw << 16) | lw) : bf16_to_f32(hw);
        pd_entry(x, bf16_to_f32((g32[q >> 1] >> sh) & 0xFFFFu), pv[q], sv[q], beta3, cs, dot, l1);
    }
    st_stream(reinterpret_cast<float4*>(t.s + j), make_float4(sv[0], sv[1], sv[2], sv[3]));
    st_stream(reinterpret_cast<float4*>(t.s + j + 4), make_float4(sv[4], sv[5], sv[6], sv[7]));
}
__device__ __forceinline__ void pd_scalar8(const PdTensor& t, const uint16_t* __restrict__ g, int64_t j, int64_t e,
                                           float beta3, float cs, float& dot, float& l1) {
    for (int q = 0; q < 8 && e + q < t.numel; ++q) {
        float sq = t.s[j + q];
        pd_entry(master(t, e + q), bf16_to_f32(g[e + q]), t.p0[j + q], sq, beta3, cs, dot, l1);
        t.s[j + q] = sq;
    }
}

// Persistent: a fixed grid (set when the group attaches) strides over the items, each thread
// taking groups of 8 consecutive entries (8 consecutive elements of one sampled block) with
// 128-bit loads when every buffer is 16-byte aligned, element by element otherwise and at a
// tensor's end.  A thread sums each item's 32 entries in fp32 and its items with compensation;
// one block reduction (double) per CTA.  slot[b]: (lr d^2 * dot, l1) of CTA b.
__global__ void __launch_bounds__(kPdThreads) k_pd_stats(const PdTensor* T, const PdItem* items,
                                                         const uint16_t* const* grads, const PdState* st,
                                                         PdStep p, double2* slots) {
    __shared__ double sm[kPdThreads / 32];
    const float df = (float)st->d;
    const double cr = ((double)p.lr * (double)df) * (double)df;
    const float cs = (float)cr;
    PdComp cdot, cl1;
    for (int b = blockIdx.x; b < p.n_items; b += gridDim.x) {
        const PdItem it = items[b];
        const PdTensor t = T[it.tensor];
        const uint16_t* __restrict__ g = grads[it.tensor];
        const bool vec = aligned16(t.w) && (t.res == nullptr || aligned16(t.res)) && aligned16(g) &&
                         aligned16(t.p0) && aligned16(t.s);
        const int64_t j0 = (int64_t)it.chunk * kPdPerCta;
        const int64_t j1 = t.len < j0 + kPdPerCta ? t.len : j0 + kPdPerCta;
        float dot = 0.f, l1 = 0.f;
#pragma unroll
        for (int i = 0; i < kPdPerThread / 8; i += 2) {
            const int64_t ja = j0 + 8 * ((int64_t)threadIdx.x + (int64_t)i * kPdThreads), jb = ja + 8 * kPdThreads;
            const int64_t ea = sampled_element(ja, p.slice_p), eb = sampled_element(jb, p.slice_p);
            const bool va = ja < j1 && vec && ea + 8 <= t.numel, vb = jb < j1 && vec && eb + 8 <= t.numel;
            Pd8 A, B;
            if (va) pd_load8(t, g, ja, ea, A);
            if (vb) pd_load8(t, g, jb, eb, B);
            if (va) pd_comp8(t, ja, A, p.beta3, cs, dot, l1);
            else if (ja < j1) pd_scalar8(t, g, ja, ea, p.beta3, cs, dot, l1);
            if (vb) pd_comp8(t, jb, B, p.beta3, cs, dot, l1);
            else if (jb < j1) pd_scalar8(t, g, jb, eb, p.beta3, cs, dot, l1);
        }
        cdot.add(dot);
        cl1.add(l1);
    }
    const double bd = block_sum_f64<kPdThreads>((double)cdot.value(), sm);
    const double bl = block_sum_f64<kPdThreads>((double)cl1.value(), sm);
    if (threadIdx.x == 0) slots[blockIdx.x] = make_double2(cr * bd, bl);
}

// One CTA: sums every slot in a fixed order into out = (sum lr d^2 dot, sum |s|) and clears them.
__global__ void __launch_bounds__(kPdEndThreads) k_pd_reduce(double2* slots, int64_t n, double* out) {
    __shared__ double sm[kPdEndThreads / 32];
    double a = 0.0, b = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += kPdEndThreads) {
        const double2 v = slots[i];
        a += v.x;
        b += v.y;
        slots[i] = make_double2(0.0, 0.0);
    }
    const double cdot = block_sum_f64<kPdEndThreads>(a, sm);
    const double l1 = block_sum_f64<kPdEndThreads>(b, sm);
    if (threadIdx.x == 0) {
        out[0] = cdot;
        out[1] = l1;
    }
}

// One thread: r and d from the step's totals.
__global__ void k_pd_finish(PdState* st, const double* total, double beta3) {
    const double r = beta3 * st->r + total[0];
    double d = st->d;
    if (total[1] > 0.0) {
        const double dhat = r / total[1];
        if (dhat > d) d = dhat;
    }
    st->r = r;
    st->d = d;
}

}  // namespace

struct ProdigyAttach {
    optim_prodigy* pd = nullptr;
    PdTensor* d_tensors = nullptr;
    PdItem* d_items = nullptr;
    FactoredDevScalars* d_kdev = nullptr;
    int32_t n_items = 0;
    cudaStream_t stream = nullptr;     // the statistics kernel's own stream
    cudaEvent_t start_ev = nullptr, done_ev = nullptr;
    int64_t slot_off = 0;
    int64_t n_slots = 0;   // CTAs of the statistics kernel (persistent grid, at least 1)
};

}  // namespace lmo

struct optim_prodigy {
    int device = 0;
    double d0 = 0.0;
    float beta3 = 0.f;
    int32_t slice_p = 1;
    lmo::PdState* d_state = nullptr;
    double* d_total = nullptr;   // this process's sums of a step (end_step's reduce/finish buffer)
    double2* d_slots = nullptr;
    int64_t n_slots = 0;
    int32_t attached = 0;
};

using namespace lmo;

namespace lmo {

void prodigy_detach(optim_group* g) {
    ProdigyAttach* a = g->prodigy;
    if (!a) return;
    if (a->pd) a->pd->attached -= 1;
    if (a->stream) cudaStreamSynchronize(a->stream);
    if (a->start_ev) cudaEventDestroy(a->start_ev);
    if (a->done_ev) cudaEventDestroy(a->done_ev);
    if (a->stream) cudaStreamDestroy(a->stream);
    cudaFree(a->d_tensors);
    cudaFree(a->d_items);
    cudaFree(a->d_kdev);
    delete a;
    g->prodigy = nullptr;
}

int prodigy_step_begin(optim_group* g, const optim_factored_hparams_t* hp, cudaStream_t s,
                       const FactoredDevScalars** kdev, cudaEvent_t* done) {
    ProdigyAttach* a = g->prodigy;
    optim_prodigy* pd = a->pd;
    PdStep p{hp->lr, hp->beta2, hp->weight_decay, pd->beta3, pd->slice_p, a->n_items};
    k_pd_scalars<<<1, 1, 0, s>>>(pd->d_state, p, a->d_kdev);
    int rc = check_cuda(cudaGetLastError(), "prodigy scalars launch");
    if (!rc) rc = check_cuda(cudaEventRecord(a->start_ev, s), "prodigy fork");
    if (!rc) rc = check_cuda(cudaStreamWaitEvent(a->stream, a->start_ev, 0), "prodigy fork");
    if (rc) return rc;
    k_pd_stats<<<(unsigned)a->n_slots, kPdThreads, 0, a->stream>>>(a->d_tensors, a->d_items, g->d_grads, pd->d_state,
                                                                   p, pd->d_slots + a->slot_off);
    rc = check_cuda(cudaGetLastError(), "prodigy statistics launch");
    // recorded even after a failed launch, so that waiting on it never waits on a stale step
    const int r2 = check_cuda(cudaEventRecord(a->done_ev, a->stream), "prodigy statistics event");
    *kdev = a->d_kdev;
    *done = a->done_ev;
    return rc ? rc : r2;
}

int prodigy_step_join(optim_group* g, cudaStream_t s) {
    return check_cuda(cudaStreamWaitEvent(s, g->prodigy->done_ev, 0), "prodigy join");
}

}  // namespace lmo

int64_t optim_prodigy_slice_len(int64_t numel, int32_t slice_p) {
    if (numel < 0 || slice_p < 1) return -1;
    const int64_t blocks = (numel + 63) / 64;
    return 64 * ((blocks + slice_p - 1) / slice_p);
}

int optim_prodigy_create(double d0, float beta3, int32_t slice_p, optim_prodigy_t** out) {
    if (!out) return set_error(OPTIM_EINVAL, "out is NULL");
    *out = nullptr;
    if (!(d0 > 0.0) || !std::isfinite(d0) || !(beta3 >= 0.0f && beta3 < 1.0f) || slice_p < 1)
        return set_error(OPTIM_EINVAL, "need d0 > 0, 0 <= beta3 < 1 and slice_p >= 1");
    optim_prodigy* pd = new optim_prodigy();
    pd->d0 = d0;
    pd->beta3 = beta3;
    pd->slice_p = slice_p;
    int rc = check_cuda(cudaGetDevice(&pd->device), "cudaGetDevice");
    if (!rc && (cudaMalloc(reinterpret_cast<void**>(&pd->d_state), sizeof(PdState)) != cudaSuccess ||
                cudaMalloc(reinterpret_cast<void**>(&pd->d_total), 2 * sizeof(double)) != cudaSuccess)) {
        cudaGetLastError();
        rc = set_error(OPTIM_ENOMEM, "prodigy state allocation failed");
    }
    if (!rc) {
        const PdState init{d0, 0.0};
        rc = check_cuda(cudaMemcpy(pd->d_state, &init, sizeof(init), cudaMemcpyHostToDevice), "prodigy state init");
    }
    if (rc) {
        cudaFree(pd->d_state);
        cudaFree(pd->d_total);
        delete pd;
        return rc;
    }
    *out = pd;
    return OPTIM_OK;
}

int optim_prodigy_destroy(optim_prodigy_t* pd) {
    if (!pd) return set_error(OPTIM_EINVAL, "controller is NULL");
    if (pd->attached > 0) return set_error(OPTIM_ESTATE, "%d groups are still attached", pd->attached);
    cudaFree(pd->d_state);
    cudaFree(pd->d_total);
    cudaFree(pd->d_slots);
    delete pd;
    return OPTIM_OK;
}

int optim_group_attach_prodigy(optim_group_t* g, optim_prodigy_t* pd, void* const* p0, void* const* s,
                               int32_t snapshot, void* stream) {
    if (!g || !pd || !p0 || !s) return set_error(OPTIM_EINVAL, "group, controller, p0 or s is NULL");
    if (snapshot != 0 && snapshot != 1) return set_error(OPTIM_EINVAL, "snapshot must be 0 or 1");
    if (g->kind != OPTIM_KIND_FACTORED) return set_error(OPTIM_EINVAL, "not a FACTORED group");
    if (g->prodigy) return set_error(OPTIM_ESTATE, "group is already attached to a controller");
    int dev = -1;
    int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev != g->device || dev != pd->device)
        return set_error(OPTIM_EINVAL, "group, controller and current device differ");
    std::vector<PdTensor> ts(g->n);
    std::vector<PdItem> items;
    for (int32_t i = 0; i < g->n; ++i) {
        const optim_tensor_desc_t& d = g->desc[i];
        if (!p0[i] || !s[i] || !is_aligned(p0[i], 4) || !is_aligned(s[i], 4))
            return set_error(OPTIM_EALIGN, "tensor %d: p0 and s must be non-NULL and 4-byte aligned", i);
        ts[i] = PdTensor{static_cast<const uint16_t*>(d.w_bf16), static_cast<const uint16_t*>(d.res_u16),
                         static_cast<float*>(p0[i]), static_cast<float*>(s[i]), d.numel,
                         optim_prodigy_slice_len(d.numel, pd->slice_p)};
        const int64_t chunks = (ts[i].len + kPdPerCta - 1) / kPdPerCta;
        for (int64_t c = 0; c < chunks; ++c) items.push_back(PdItem{i, (int32_t)c});
    }
    if (items.size() > (size_t)INT32_MAX / 2) return set_error(OPTIM_EINVAL, "too many statistics blocks");
    ProdigyAttach* a = new ProdigyAttach();
    a->pd = pd;
    a->n_items = (int32_t)items.size();
    const int per_sm = pd->slice_p >= 4 ? kPdCtasPerSmSparse : kPdCtasPerSmDense;
    const int64_t grid = std::min<int64_t>(a->n_items, (int64_t)per_sm * sm_count());
    a->n_slots = grid > 0 ? grid : 1;
    auto fail = [&](int code) {
        if (a->start_ev) cudaEventDestroy(a->start_ev);
        if (a->done_ev) cudaEventDestroy(a->done_ev);
        if (a->stream) cudaStreamDestroy(a->stream);
        cudaFree(a->d_tensors);
        cudaFree(a->d_items);
        cudaFree(a->d_kdev);
        delete a;
        return code;
    };
    if (cudaMalloc(reinterpret_cast<void**>(&a->d_tensors), ts.size() * sizeof(PdTensor) + 1) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&a->d_items), items.size() * sizeof(PdItem) + 1) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&a->d_kdev), sizeof(FactoredDevScalars)) != cudaSuccess) {
        cudaGetLastError();
        return fail(set_error(OPTIM_ENOMEM, "prodigy table allocation failed"));
    }
    rc = check_cuda(cudaStreamCreateWithFlags(&a->stream, cudaStreamNonBlocking), "prodigy stream");
    if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&a->start_ev, cudaEventDisableTiming), "prodigy event");
    if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&a->done_ev, cudaEventDisableTiming), "prodigy event");
    if (rc) return fail(rc);
    // grow the controller's slot array (between steps: the device is idle after the sync)
    rc = check_cuda(cudaDeviceSynchronize(), "device synchronize");
    double2* slots = nullptr;
    if (!rc && cudaMalloc(reinterpret_cast<void**>(&slots), (size_t)(pd->n_slots + a->n_slots) * sizeof(double2)) != cudaSuccess) {
        cudaGetLastError();
        rc = set_error(OPTIM_ENOMEM, "prodigy slot allocation failed");
    }
    if (!rc) rc = check_cuda(cudaMemset(slots, 0, (size_t)(pd->n_slots + a->n_slots) * sizeof(double2)), "slot clear");
    if (!rc && pd->n_slots > 0)
        rc = check_cuda(cudaMemcpy(slots, pd->d_slots, (size_t)pd->n_slots * sizeof(double2), cudaMemcpyDeviceToDevice),
                        "slot copy");
    if (!rc && !ts.empty())
        rc = check_cuda(cudaMemcpy(a->d_tensors, ts.data(), ts.size() * sizeof(PdTensor), cudaMemcpyHostToDevice), "table upload");
    if (!rc && !items.empty())
        rc = check_cuda(cudaMemcpy(a->d_items, items.data(), items.size() * sizeof(PdItem), cudaMemcpyHostToDevice), "table upload");
    if (rc) {
        cudaFree(slots);
        return fail(rc);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (snapshot && a->n_items > 0) {
        k_pd_snapshot<<<(unsigned)a->n_items, kPdThreads, 0, st>>>(a->d_tensors, a->d_items, pd->slice_p);
        rc = check_cuda(cudaGetLastError(), "prodigy snapshot launch");
        if (rc) {
            cudaFree(slots);
            return fail(rc);
        }
    }
    cudaFree(pd->d_slots);
    pd->d_slots = slots;
    a->slot_off = pd->n_slots;
    pd->n_slots += a->n_slots;
    pd->attached += 1;
    g->prodigy = a;
    return OPTIM_OK;
}

int optim_prodigy_reduce(optim_prodigy_t* pd, double* partial, void* stream) {
    if (!pd || !partial) return set_error(OPTIM_EINVAL, "controller or partial is NULL");
    if (!is_aligned(partial, 8)) return set_error(OPTIM_EALIGN, "partial must be 8-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pd->n_slots == 0) return check_cuda(cudaMemsetAsync(partial, 0, 2 * sizeof(double), st), "partial clear");
    k_pd_reduce<<<1, kPdEndThreads, 0, st>>>(pd->d_slots, pd->n_slots, partial);
    return check_cuda(cudaGetLastError(), "prodigy reduce launch");
}

int optim_prodigy_finish(optim_prodigy_t* pd, const double* total, void* stream) {
    if (!pd || !total) return set_error(OPTIM_EINVAL, "controller or total is NULL");
    if (!is_aligned(total, 8)) return set_error(OPTIM_EALIGN, "total must be 8-byte aligned");
    k_pd_finish<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(pd->d_state, total, (double)pd->beta3);
    return check_cuda(cudaGetLastError(), "prodigy finish launch");
}

int optim_prodigy_end_step(optim_prodigy_t* pd, void* stream) {
    if (!pd) return set_error(OPTIM_EINVAL, "controller is NULL");
    int rc = optim_prodigy_reduce(pd, pd->d_total, stream);
    if (!rc) rc = optim_prodigy_finish(pd, pd->d_total, stream);
    return rc;
}

int optim_prodigy_get(optim_prodigy_t* pd, double* d, double* r) {
    if (!pd || !d || !r) return set_error(OPTIM_EINVAL, "controller, d or r is NULL");
    PdState h{};
    int rc = check_cuda(cudaDeviceSynchronize(), "device synchronize");
    if (!rc) rc = check_cuda(cudaMemcpy(&h, pd->d_state, sizeof(h), cudaMemcpyDeviceToHost), "prodigy state read");
    if (rc) return rc;
    *d = h.d;
    *r = h.r;
    return OPTIM_OK;
}

int optim_prodigy_set(optim_prodigy_t* pd, double d, double r) {
    if (!pd) return set_error(OPTIM_EINVAL, "controller is NULL");
    if (!(d > 0.0) || !std::isfinite(d) || !std::isfinite(r)) return set_error(OPTIM_EINVAL, "need d > 0 and finite r");
    const PdState h{d, r};
    int rc = check_cuda(cudaDeviceSynchronize(), "device synchronize");
    if (!rc) rc = check_cuda(cudaMemcpy(pd->d_state, &h, sizeof(h), cudaMemcpyHostToDevice), "prodigy state write");
    return rc;
}
