// factored.cu -- factored second-moment step (Adafactor / Prodigy, beta1 = 0, no exp_avg).
//
// Follows the printed fused Adafactor step ("Fused backward pass" commit,
// library/adafactor_fused.py, adafactor_step_param) with a fixed learning rate and the eps2
// placement of prodigy PR #25 ("more VRAM savings: no first moment and factored second moment"):
//   q = g*g + eps1 (Adafactor) | g*g (Prodigy)
//   R = b2t*R + alpha*mean_j(q) (+eps2),  C = b2t*C + alpha*mean_i(q) (+eps2)
//   u_ij = (rsqrt(R_i / mean(R)) * rsqrt(C_j)) * g_ij        (1-D: u = rsqrt(V) * g);  Prodigy: u = u * d
//   u = (u / max(1, RMS(u)/clip)) * lr_eff;  w = w + w*(-wd*lr_eff);  w = w - u;  Kahan split
// Factoring is over the last two dims; leading dims are a batch of matrices.
//
// Tensor classes and their kernels:
//   wide  (ndim >= 2, rows*cols > 16): 128x256 tiles, 256 threads (8 warps x 16 rows, lane = 8 cols)
//   tiny  (ndim >= 2, rows*cols <= 16, e.g. 3x3 conv kernels): 2048 matrices per CTA, staged
//         through shared memory in sub-batches of 256 (64 for shapes beyond 9 elements or 6
//         statistics), one thread per matrix, cp.async double buffering
//   vector (ndim == 1): one thread per element, full fp32 second moment
// Per wave of tensors (waves keep the wave's gradients, read three times, within L2):
//   1. k_stats  : wide tiles -> row/column partial sums of q;  tiny/vector -> state EMA, u, sum u^2
//   2. k_final  : wide matrices -> R EMA over 256-row blocks (mean(R) by the last block of a
//                 matrix), C EMA over 64-column blocks, rsqrt factor per column
//   3. k_rms    : wide tiles -> sum u^2 per tile
//   4. k_apply  : every element -> clip, lr, decay, subtract, split
// The clip divisor of a tensor is computed by the last CTA to finish its partial sums (threadfence
// and counter), summing the partials in a fixed order.  Every reduction is in a fixed order, so
// results are deterministic; sums are fp32 trees, with compensated (Neumaier) sums across partials.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "factored.h"

namespace lmo {

namespace {

constexpr int kTR = 128;     // rows per wide tile (16 per warp, in two batches of eight)
constexpr int kTC = 256;     // columns per wide tile
constexpr int kFinRowsPerItem = 256;   // rows per finalize row block (one per thread)
constexpr int kFinColsPerItem = 32;    // columns per finalize column block
constexpr int kFinGroups = kThreads / kFinColsPerItem;   // band groups of a column block (8)
constexpr int kTinySub = kThreads;     // small matrices per staged sub-batch (one per thread)
constexpr int kTinyPerCta = 8 * kTinySub;
constexpr int kVecPerCta = kThreads * 8;
// Gradient bytes per wave (the L2-resident target) and the number of waves in flight at once
// (the caller's stream plus kWaveStreams - 1 internal streams).
#ifndef LMOPT_WAVE_MB
#define LMOPT_WAVE_MB 96
#endif
#ifndef LMOPT_WAVE_STREAMS
#define LMOPT_WAVE_STREAMS 3
#endif
constexpr int64_t kWaveGradBytes = (int64_t)LMOPT_WAVE_MB << 20;
constexpr int kWaveStreams = LMOPT_WAVE_STREAMS;

enum : int32_t { kWide = 0, kTiny = 1, kVec = 2 };
enum : int32_t { kFinRows = 0, kFinCols = 1 };

struct FTensor {
    uint16_t* w;
    uint16_t* res;
    float* row;     // R state [B*R] (wide, tiny)
    float* col;     // C state [B*C] (wide, tiny) or V [numel] (vector)
    int64_t numel;
    int64_t B, R, C;
    int32_t cls;
    int32_t ncb;    // column blocks (wide)
    int32_t nbands; // row bands (wide)
    int32_t ss_cnt;
    int32_t n_rowitems;  // finalize row blocks per matrix (wide)
    int32_t pad;
    int64_t rowpart_off, colpart_off, cc_off, ss_off;
    int64_t mat_off;     // first matrix index of this tensor (mean(R) and its counter)
    int64_t rbarpart_off;
};

struct Item {        // one CTA of k_stats / k_rms / k_apply / k_final
    int32_t tensor;
    int32_t cls;     // kWide / kTiny / kVec (k_final: kFinRows / kFinCols)
    int32_t x;       // wide: matrix; tiny: first matrix; vector: chunk; final: matrix
    int32_t band;    // wide: row band
    int32_t cb;      // wide: 256-column block; final: row block / 64-column block
    int32_t part;    // index of this CTA's sum-of-squares partial within its tensor
};

struct Dev {
    const FTensor* tensors;
    const uint16_t* const* grads;
    float* rowpart;
    float* colpart;
    float* cc;
    float* rbar;        // mean(R) per matrix
    float* rbarpart;    // per finalize row block
    float* ss;
    float* den;
    unsigned* counter;  // per tensor (sum of squares)
    unsigned* rcounter; // per matrix (mean of R)
    unsigned long long* nonfinite;   // CTAs of the update that stored a non-finite weight (or null)
};

struct K {
    float b2t, alpha, eps1, eps2, clip, lr_eff, nwdlr;
    int32_t mode;
    float unum;
    const FactoredDevScalars* kdev;
};
// The d-dependent scalars from device memory when d is adaptive; called by every kernel right
// after its programmatic-launch wait, so that the statistics kernel that wrote them is complete.
__device__ __forceinline__ void load_k(K& k) {
    if (k.kdev == nullptr) return;
    const FactoredDevScalars v = *k.kdev;
    k.alpha = v.alpha;
    k.lr_eff = v.lr_eff;
    k.nwdlr = v.nwdlr;
    k.unum = v.unum;
}

__device__ __forceinline__ float qval(float g, const K& k) {
    float gg = __fmul_rn(g, g);
    return k.mode == 0 ? __fadd_rn(gg, k.eps1) : gg;
}
__device__ __forceinline__ float ema(float s, float x, const K& k) {
    float r = __fadd_rn(__fmul_rn(k.b2t, s), __fmul_rn(k.alpha, x));
    return k.mode == 1 ? __fadd_rn(r, k.eps2) : r;
}
// 1/sqrt(x) rounded once (correctly rounded reciprocal square root).
__device__ __forceinline__ float rsqrt_rn(float x) { return __frsqrt_rn(x); }
// Columns of a lane's 8-column group that lie inside the matrix (0..8).
__device__ __forceinline__ int cols_in(int64_t remaining) {
    return remaining <= 0 ? 0 : (remaining >= 8 ? 8 : (int)remaining);
}

// L2 eviction priority of the gradient loads: the statistics and RMS kernels keep a wave's
// gradients (read again by the next kernels) ahead of streaming data; the update kernel, their
// last reader, marks them first to go.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_keep(const uint4* a, uint64_t pol) {
    uint4 v;
    asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(a), "l"(pol));
    return v;
}

// Neumaier-compensated accumulation.
struct Comp {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        float t = __fadd_rn(s, x);
        if (fabsf(s) >= fabsf(x)) c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), x));
        else c = __fadd_rn(c, __fadd_rn(__fsub_rn(x, t), s));
        s = t;
    }
    __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

// Programmatic dependent launch.  The four kernels of a wave are launched so that each may
// start while its predecessor on the stream drains.  pdl_wait blocks (in hardware) until the
// predecessor grid has completed and its writes are visible; before it a kernel only reads what
// no kernel of the step writes (its work items, the tensor table, gradients, and in the update
// kernel the weight words, which only that kernel writes).  Every kernel signals its dependents
// only after its own wait, so a kernel that starts early can rely on everything before its
// predecessor having completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_sync() {
    pdl_wait();
    pdl_release();
}

// Block-wide fp32 sum in a fixed tree; result valid in every thread.
__device__ float block_sum(float x, float* sm /* 32 floats */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum_f32(x);
    __syncthreads();
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    float y = lane < (int)(blockDim.x >> 5) ? sm[lane] : 0.f;
    y = warp_sum_f32(y);
    return y;
}

// Counts this CTA once if any of its threads stored a non-finite weight (nf: the largest bf16
// magnitude a thread stored; 0x7F80 and above is infinity or NaN).  Every thread of the CTA calls
// it once (a barrier).
__device__ __forceinline__ void count_nonfinite(const Dev& D, uint32_t nf) {
    const int any = __syncthreads_or(nf >= 0x7F80u);
    if (any && threadIdx.x == 0 && D.nonfinite) atomicAdd(D.nonfinite, 1ull);
}
__device__ __forceinline__ uint32_t max_bf16_mag(uint32_t nf, const uint4& W) {
    uint32_t x = __vmaxu2(__vmaxu2(W.x & 0x7FFF7FFFu, W.y & 0x7FFF7FFFu), __vmaxu2(W.z & 0x7FFF7FFFu, W.w & 0x7FFF7FFFu));
    return max(nf, max(x & 0xFFFFu, x >> 16));
}

// Per-tensor update scale: lr when the update is not clipped (den == 1), else fl(lr / den).  The
// clipped update is then fl(u * fl(lr / den)) rather than fl(fl(u / den) * lr): one multiply per
// element instead of a division, within about one ulp of the update.
__device__ __forceinline__ float update_scale(float den, const K& k) {
    return den == 1.0f ? k.lr_eff : __fdiv_rn(k.lr_eff, den);
}
// The update's numerator factor: u d in Prodigy mode (the first moment of Prodigy with beta1 = 0
// is d g), applied to each element before its square is summed and before the clip, as the
// step is defined; Adafactor mode leaves u as it is.
template <bool kP>
__device__ __forceinline__ float numer(float u, const K& k) { return kP ? __fmul_rn(u, k.unum) : u; }
__device__ __forceinline__ float numer_rt(float u, const K& k) { return k.mode == 1 ? __fmul_rn(u, k.unum) : u; }

__device__ __forceinline__ void apply_elem(uint32_t& hi, uint32_t& lo, bool has_res, float u, float s, const K& k) {
    float w = has_res ? __uint_as_float((hi << 16) | lo) : bf16_to_f32(hi);
    const float uu = __fmul_rn(u, s);
    if (k.nwdlr != 0.0f) w = __fadd_rn(w, __fmul_rn(w, k.nwdlr));
    w = __fsub_rn(w, uu);
    const uint32_t b = __float_as_uint(w);
    if (has_res) {
        hi = b >> 16;
        lo = b & 0xFFFFu;
    } else {
        hi = rne_bf16(w);
    }
}

// Clip divisor from the tensor's fp32 sum of squares of the update (numerator factor included).
__device__ __forceinline__ float clip_den(float ss, int64_t n, float clip) {
    const float ms = __fdiv_rn(ss, (float)n);
    const float r = __fdiv_rn(__fsqrt_rn(ms), clip);
    return r < 1.0f ? 1.0f : r;   // a NaN RMS stays NaN (clamp(min=1) semantics), as in the oracle
}

// Writes this CTA's partial; the last CTA of the tensor sums all partials (fixed order) and
// writes the clip divisor.  Must be called by every thread of the CTA.
__device__ void finish_ss(const Dev& D, const FTensor& t, int tensor, int part, float block_total,
                          const K& k, float* sm) {
    __shared__ bool last;
    if (threadIdx.x == 0) {
        D.ss[t.ss_off + part] = block_total;
        __threadfence();
        const unsigned prev = atomicAdd(&D.counter[tensor], 1u);
        last = prev == (unsigned)t.ss_cnt - 1u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    Comp acc;
    for (int i = threadIdx.x; i < t.ss_cnt; i += blockDim.x) acc.add(__ldcg(D.ss + t.ss_off + i));
    const float tot = block_sum(acc.value(), sm);
    if (threadIdx.x == 0) {
        D.den[tensor] = clip_den(tot, t.numel, k.clip);
        D.counter[tensor] = 0u;
    }
}

// Loads 8 consecutive bf16 words (columns col0..col0+7 of one row) into v[8]; columns past
// `ncols` read as 0.
__device__ __forceinline__ void load8(const uint16_t* p, int ncols, uint32_t (&v)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < ncols ? p[j] : 0u;
}

// Copies n elements from global to shared memory (or back), 128 bits at a time when both sides
// are 16-byte aligned and the byte count is a multiple of 16.  Called by the whole CTA.
template <class T>
__device__ __forceinline__ void stage(T* dst, const T* src, int n) {
    if (aligned16(src) && aligned16(dst) && ((n * (int)sizeof(T)) & 15) == 0) {
        const int nv = n * (int)sizeof(T) / 16;
        for (int i = threadIdx.x; i < nv; i += blockDim.x)
            reinterpret_cast<uint4*>(dst)[i] = __ldcg(reinterpret_cast<const uint4*>(src) + i);
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
    }
}
template <class T>
__device__ __forceinline__ void unstage(T* dst, const T* src, int n, bool streaming) {
    if (aligned16(src) && aligned16(dst) && ((n * (int)sizeof(T)) & 15) == 0) {
        const int nv = n * (int)sizeof(T) / 16;
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            const uint4 x = reinterpret_cast<const uint4*>(src)[i];
            if (streaming) st_stream(reinterpret_cast<uint4*>(dst) + i, x);
            else reinterpret_cast<uint4*>(dst)[i] = x;
        }
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
    }
}

// Shared-memory staging of the small-matrix class, two buffers (double buffering).  A buffer
// holds one sub-batch: gradient / weight / residual words and the R then C statistics.  It is
// sized for kTinySub matrices of up to 9 words and 6 statistics (3x3, 1x1, 2x2, 2x4 ...); other
// small shapes (rows*cols <= 16, hence rows + cols <= 17) take sub-batches of kTinySub / 4.
constexpr int kTinyWords = kTinySub * 9;    // u16 words per word plane per buffer
constexpr int kTinyStats = kTinySub * 6;    // floats per buffer
static_assert((kTinySub / 4) * 16 <= kTinyWords && (kTinySub / 4) * 17 <= kTinyStats, "small sub-batch must fit");
constexpr int kStatsSmem = 2 * (kTinyWords * 2 + kTinyStats * 4);
constexpr int kApplySmem = 2 * (3 * kTinyWords * 2 + kTinyStats * 4);
static_assert(kStatsSmem >= 8 * (kTC + 1) * 4, "wide column buffer must fit the shared area");
static_assert((kTinyWords * 2) % 16 == 0 && (kTinyStats * 4) % 16 == 0, "buffers must stay 16-byte aligned");

__device__ __forceinline__ int tiny_sub(int r, int c) { return (r * c <= 9 && r + c <= 6) ? kTinySub : kTinySub / 4; }

// Asynchronous 16-byte global -> shared copies (cp.async, completion tracked per thread by
// commit groups; the hardware wait needs no polling loop).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
// `bytes` a multiple of 16, both addresses 16-byte aligned.
__device__ __forceinline__ void stage_async(void* dst, const void* src, int bytes) {
    for (int i = threadIdx.x; i < (bytes >> 4); i += blockDim.x)
        cp_async16(static_cast<char*>(dst) + 16 * i, static_cast<const char*>(src) + 16 * i);
}

// Any small matrix (rows*cols <= 16): R, C EMAs (written back), mean(R), and the matrix's sum of
// squared updates.
__device__ __noinline__ float tiny_stats_any(const uint16_t* gm, float* Rs, float* Cs, int r, int c, const K& k) {
    float q[16], rsum[16], csum[16];
    for (int e = 0; e < r * c; ++e) q[e] = qval(bf16_to_f32(gm[e]), k);
    float rtot = 0.f;
    for (int i = 0; i < r; ++i) {
        float s = 0.f;
        for (int j = 0; j < c; ++j) s = __fadd_rn(s, q[i * c + j]);
        const float nr = ema(Rs[i], __fdiv_rn(s, (float)c), k);
        Rs[i] = nr;
        rsum[i] = nr;
        rtot = __fadd_rn(rtot, nr);
    }
    for (int j = 0; j < c; ++j) {
        float s = 0.f;
        for (int i = 0; i < r; ++i) s = __fadd_rn(s, q[i * c + j]);
        const float nc = ema(Cs[j], __fdiv_rn(s, (float)r), k);
        Cs[j] = nc;
        csum[j] = rsqrt_rn(nc);
    }
    const float rbar = __fdiv_rn(rtot, (float)r);
    float acc = 0.f;
    for (int i = 0; i < r; ++i) {
        const float rr = rsqrt_rn(__fdiv_rn(rsum[i], rbar));
        for (int j = 0; j < c; ++j) {
            const float u = numer_rt(__fmul_rn(__fmul_rn(rr, csum[j]), bf16_to_f32(gm[i * c + j])), k);
            acc = __fadd_rn(acc, __fmul_rn(u, u));
        }
    }
    return acc;
}

// 3x3 matrices (the convolution kernels) with the per-tensor switches as template parameters:
// Prodigy mode (eps2 after the EMA), a residual, decoupled decay.  The factors use the hardware
// reciprocal square root rsqrtf (at most 2 ulp from 1/sqrt, CUDA's documented bound), the means
// products with fl(1/3), so the per-matrix work is a few dozen instructions; both kernels compute
// the factors the same way.
struct Fac3 {
    float rr[3], cc[3];
};
__device__ __forceinline__ Fac3 factors3(float r0, float r1, float r2, const float* Cs) {
    Fac3 f;
    const float inv_rbar = __frcp_rn(__fmul_rn(__fadd_rn(__fadd_rn(r0, r1), r2), 1.0f / 3.0f));
    f.rr[0] = rsqrtf(__fmul_rn(r0, inv_rbar));
    f.rr[1] = rsqrtf(__fmul_rn(r1, inv_rbar));
    f.rr[2] = rsqrtf(__fmul_rn(r2, inv_rbar));
    f.cc[0] = rsqrtf(Cs[0]);
    f.cc[1] = rsqrtf(Cs[1]);
    f.cc[2] = rsqrtf(Cs[2]);
    return f;
}
template <bool kProdigy>
__device__ __forceinline__ float stats3(const uint16_t* gm, float* Rs, float* Cs, const K& k) {
    float q[9];
#pragma unroll
    for (int e = 0; e < 9; ++e) {
        const float g = bf16_to_f32(gm[e]);
        q[e] = kProdigy ? __fmul_rn(g, g) : __fadd_rn(__fmul_rn(g, g), k.eps1);
    }
    float nr[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const float s = __fadd_rn(__fadd_rn(q[3 * i], q[3 * i + 1]), q[3 * i + 2]);
        float v = __fadd_rn(__fmul_rn(k.b2t, Rs[i]), __fmul_rn(k.alpha, __fmul_rn(s, 1.0f / 3.0f)));
        if (kProdigy) v = __fadd_rn(v, k.eps2);
        Rs[i] = v;
        nr[i] = v;
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const float s = __fadd_rn(__fadd_rn(q[j], q[3 + j]), q[6 + j]);
        float v = __fadd_rn(__fmul_rn(k.b2t, Cs[j]), __fmul_rn(k.alpha, __fmul_rn(s, 1.0f / 3.0f)));
        if (kProdigy) v = __fadd_rn(v, k.eps2);
        Cs[j] = v;
    }
    const Fac3 f = factors3(nr[0], nr[1], nr[2], Cs);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 9; ++e) {
        float u = __fmul_rn(__fmul_rn(f.rr[e / 3], f.cc[e % 3]), bf16_to_f32(gm[e]));
        if (kProdigy) u = __fmul_rn(u, k.unum);
        acc = __fmaf_rn(u, u, acc);
    }
    return acc;
}
template <bool kRes, bool kDecay, bool kProdigy>
__device__ __forceinline__ void apply3(uint16_t* wm, uint16_t* rm, const uint16_t* gm, const float* Rs,
                                       const float* Cs, float us, float nwdlr, float unum) {
    const Fac3 f = factors3(Rs[0], Rs[1], Rs[2], Cs);
#pragma unroll
    for (int e = 0; e < 9; ++e) {
        float w = kRes ? __uint_as_float(((uint32_t)wm[e] << 16) | rm[e]) : bf16_to_f32(wm[e]);
        float u = __fmul_rn(__fmul_rn(f.rr[e / 3], f.cc[e % 3]), bf16_to_f32(gm[e]));
        if (kProdigy) u = __fmul_rn(u, unum);
        if (kDecay) w = __fadd_rn(w, __fmul_rn(w, nwdlr));
        w = __fsub_rn(w, __fmul_rn(u, us));
        const uint32_t b = __float_as_uint(w);
        if (kRes) {
            wm[e] = (uint16_t)(b >> 16);
            rm[e] = (uint16_t)(b & 0xFFFFu);
        } else {
            wm[e] = (uint16_t)rne_bf16(w);
        }
    }
}

// 3x3 tensors whose every sub-batch is whole and whose buffers are 16-byte aligned (the
// convolution kernels): the staging loops have compile-time trip counts.  Per sub-batch of
// kTinySub matrices: 288 gradient (weight, residual) chunks of 16 bytes, 192 R and 192 C chunks.
constexpr int k3Words = kTinySub * 9 * 2 / 16;   // 16-byte chunks of one word plane
constexpr int k3Stats = kTinySub * 3 * 4 / 16;   // 16-byte chunks of R (and of C)
static_assert(k3Words > kTinySub && k3Words <= 2 * kTinySub && k3Stats <= kTinySub, "chunk counts per thread");

template <bool kProdigy>
__device__ __forceinline__ float conv3_stats(const uint16_t* g, float* row, float* col, int64_t m_first, int nsub,
                                             unsigned char* smem, const K& k) {
    const int tid = threadIdx.x;
    auto gbuf = [&](int b) { return reinterpret_cast<uint4*>(smem + b * (kTinyWords * 2)); };
    auto sbuf = [&](int b) { return reinterpret_cast<uint4*>(smem + 2 * kTinyWords * 2 + b * (kTinyStats * 4)); };
    auto issue = [&](int kk) {
        const int64_t m = m_first + (int64_t)kk * kTinySub;
        const uint4* gs = reinterpret_cast<const uint4*>(g + m * 9);
        const uint4* rs = reinterpret_cast<const uint4*>(row + m * 3);
        const uint4* cs = reinterpret_cast<const uint4*>(col + m * 3);
        uint4* gd = gbuf(kk & 1);
        uint4* sd = sbuf(kk & 1);
        cp_async16(gd + tid, gs + tid);
        if (tid < k3Words - kTinySub) cp_async16(gd + kTinySub + tid, gs + kTinySub + tid);
        if (tid < k3Stats) {
            cp_async16(sd + tid, rs + tid);
            cp_async16(sd + k3Stats + tid, cs + tid);
        }
        cp_async_commit();
    };
    float acc = 0.f;
    issue(0);
    for (int kk = 0; kk < nsub; ++kk) {
        if (kk + 1 < nsub) {
            issue(kk + 1);   // its buffer was released by the barrier ending iteration kk-1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int b = kk & 1;
        float* R = reinterpret_cast<float*>(sbuf(b));
        acc = __fadd_rn(acc, stats3<kProdigy>(reinterpret_cast<const uint16_t*>(gbuf(b)) + tid * 9, R + tid * 3,
                                              R + kTinySub * 3 + tid * 3, k));
        __syncthreads();
        const int64_t m = m_first + (int64_t)kk * kTinySub;
        if (tid < k3Stats) {
            reinterpret_cast<uint4*>(row + m * 3)[tid] = sbuf(b)[tid];
            reinterpret_cast<uint4*>(col + m * 3)[tid] = sbuf(b)[k3Stats + tid];
        }
        __syncthreads();
    }
    return acc;
}

template <bool kRes, bool kDecay, bool kProdigy>
__device__ __forceinline__ uint32_t conv3_apply(const uint16_t* g, uint16_t* w, uint16_t* res, const float* row,
                                            const float* col, int64_t m_first, int nsub, unsigned char* smem, float us,
                                            float nwdlr, float unum) {
    constexpr int kBuf = 3 * kTinyWords * 2 + kTinyStats * 4;
    const int tid = threadIdx.x;
    uint32_t nf = 0u;
    auto plane = [&](int b, int a) { return reinterpret_cast<uint4*>(smem + b * kBuf + a * (kTinyWords * 2)); };
    auto issue = [&](int kk) {
        const int64_t m = m_first + (int64_t)kk * kTinySub;
        const int b = kk & 1;
        const uint4* src[3] = {reinterpret_cast<const uint4*>(g + m * 9), reinterpret_cast<const uint4*>(w + m * 9),
                               kRes ? reinterpret_cast<const uint4*>(res + m * 9) : nullptr};
#pragma unroll
        for (int a = 0; a < (kRes ? 3 : 2); ++a) {
            cp_async16(plane(b, a) + tid, src[a] + tid);
            if (tid < k3Words - kTinySub) cp_async16(plane(b, a) + kTinySub + tid, src[a] + kTinySub + tid);
        }
        if (tid < k3Stats) {
            cp_async16(plane(b, 3) + tid, reinterpret_cast<const uint4*>(row + m * 3) + tid);
            cp_async16(plane(b, 3) + k3Stats + tid, reinterpret_cast<const uint4*>(col + m * 3) + tid);
        }
        cp_async_commit();
    };
    issue(0);
    for (int kk = 0; kk < nsub; ++kk) {
        if (kk + 1 < nsub) {
            issue(kk + 1);   // its buffer was released by the barrier ending iteration kk-1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int b = kk & 1;
        const float* R = reinterpret_cast<const float*>(plane(b, 3));
        apply3<kRes, kDecay, kProdigy>(reinterpret_cast<uint16_t*>(plane(b, 1)) + tid * 9,
                                       reinterpret_cast<uint16_t*>(plane(b, 2)) + tid * 9,
                                       reinterpret_cast<const uint16_t*>(plane(b, 0)) + tid * 9, R + tid * 3,
                                       R + kTinySub * 3 + tid * 3, us, nwdlr, unum);
        __syncthreads();
        const int64_t m = m_first + (int64_t)kk * kTinySub;
#pragma unroll
        for (int a = 1; a < (kRes ? 3 : 2); ++a) {
            uint16_t* base = a == 1 ? w : res;   // a == 2 only with a residual
            uint4* dst = reinterpret_cast<uint4*>(base + m * 9);
            const uint4 x0 = plane(b, a)[tid];
            st_stream(dst + tid, x0);
            if (a == 1) nf = max_bf16_mag(nf, x0);
            if (tid < k3Words - kTinySub) {
                const uint4 x1 = plane(b, a)[kTinySub + tid];
                st_stream(dst + kTinySub + tid, x1);
                if (a == 1) nf = max_bf16_mag(nf, x1);
            }
        }
        __syncthreads();
    }
    return nf;
}

// Statistics of one staged small matrix, out of line (the ragged / unaligned staging path).
__device__ __noinline__ float tiny_stats_call(const uint16_t* gm, float* Rs, float* Cs, int r, int c, const K& k) {
    if (r == 3 && c == 3) return k.mode == 1 ? stats3<true>(gm, Rs, Cs, k) : stats3<false>(gm, Rs, Cs, k);
    return tiny_stats_any(gm, Rs, Cs, r, c, k);
}

// Apply step of any small matrix on staged words (w, res, g and R, C in shared memory).
template <bool kP>
__device__ __noinline__ void tiny_apply_any(uint16_t* wm, uint16_t* rm, const uint16_t* gm, const float* Rs, const float* Cs,
                               int r, int c, bool has_res, float us, const K& k) {
    float rtot = 0.f, cfac[16];
    for (int i = 0; i < r; ++i) rtot = __fadd_rn(rtot, Rs[i]);
    const float rbar = __fdiv_rn(rtot, (float)r);
    for (int j = 0; j < c; ++j) cfac[j] = rsqrt_rn(Cs[j]);
    for (int i = 0; i < r; ++i) {
        const float rr = rsqrt_rn(__fdiv_rn(Rs[i], rbar));
        for (int j = 0; j < c; ++j) {
            const int e = i * c + j;
            uint32_t hi = wm[e], lo = has_res ? rm[e] : 0u;
            apply_elem(hi, lo, has_res, numer<kP>(__fmul_rn(__fmul_rn(rr, cfac[j]), bf16_to_f32(gm[e])), k), us, k);
            wm[e] = (uint16_t)hi;
            if (has_res) rm[e] = (uint16_t)lo;
        }
    }
}

// Packed fp32 pairs: __fmul2_rn / __fadd2_rn / __ffma2_rn round each component exactly as the
// scalar _rn operations, so pairing changes no result, only the instruction count.
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
// The two bf16 values of one 32-bit word as fp32 (exact), low half first.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Sums each of v[0..7] over the 32 lanes of the warp in 9 shuffles (a transposing butterfly:
// every exchange halves the number of values a lane carries).  Lanes 4r..4r+3 return the total
// of v[r]; the tree is fixed and each pairwise add is commutative, so the four copies agree.
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
    const unsigned full = 0xFFFFFFFFu;
    float a[4], b[2];
    const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = h4 ? v[i + 4] : v[i], send = h4 ? v[i] : v[i + 4];
        a[i] = __fadd_rn(keep, __shfl_xor_sync(full, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = h3 ? a[i + 2] : a[i], send = h3 ? a[i] : a[i + 2];
        b[i] = __fadd_rn(keep, __shfl_xor_sync(full, send, 8));
    }
    const float keep = h2 ? b[1] : b[0], send = h2 ? b[0] : b[1];
    float c = __fadd_rn(keep, __shfl_xor_sync(full, send, 4));
    c = __fadd_rn(c, __shfl_xor_sync(full, c, 2));
    return __fadd_rn(c, __shfl_xor_sync(full, c, 1));
}


// ------------------------------------------------------------------------------------ stats
template <bool kP>
__global__ void __launch_bounds__(kThreads, 4) k_stats(Dev D, const Item* items, K k) {
    __shared__ float sm[32];
    __shared__ __align__(16) unsigned char smem[kStatsSmem];
    const Item it = items[blockIdx.x];
    const FTensor t = D.tensors[it.tensor];
    const uint16_t* __restrict__ g = D.grads[it.tensor];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_sync();
    load_k(k);

    const uint64_t keep = l2_keep_policy();
    if (it.cls == kWide) {
        float (*cols)[kTC + 1] = reinterpret_cast<float (*)[kTC + 1]>(smem);
        const int64_t b = it.x;
        const int64_t col0 = (int64_t)it.cb * kTC + lane * 8;
        const int ncols = cols_in(t.C - col0);
        // The branch below must be the same for every lane: both sides contain full-warp
        // shuffles.  With C a multiple of 8 a lane's group is either whole (8) or empty (0).
        const bool vec = aligned16(g) && (t.C % 8 == 0);
        const bool lane_ok = ncols == 8;
        const int64_t row0 = (int64_t)it.band * kTR + warp;   // this warp's rows: row0 + 8*kk
        float cacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (vec) {
            const float eq = k.mode == 0 ? k.eps1 : 0.0f;   // + 0 leaves g*g unchanged (Prodigy mode)
            float2 c2[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
#pragma unroll 1
            for (int kb = 0; kb < kTR / 64; ++kb) {
                // eight rows' loads issued before any use (memory-level parallelism)
                uint4 x[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int64_t row = row0 + 64 * kb + 8 * kk;
                    x[kk] = (row < t.R && lane_ok)
                                ? ld_keep(reinterpret_cast<const uint4*>(g + (b * t.R + row) * t.C + col0), keep)
                                : make_uint4(0, 0, 0, 0);
                }
                float rs[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int64_t row = row0 + 64 * kb + 8 * kk;
                    rs[kk] = 0.f;
                    if (lane_ok && row < t.R) {
                        const uint32_t wd[4] = {x[kk].x, x[kk].y, x[kk].z, x[kk].w};
                        float2 r2 = f2(0.f);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 gq = bf16x2_to_f2(wd[q]);
                            const float2 qq = __fadd2_rn(__fmul2_rn(gq, gq), f2(eq));
                            r2 = __fadd2_rn(r2, qq);
                            c2[q] = __fadd2_rn(c2[q], qq);
                        }
                        rs[kk] = __fadd_rn(r2.x, r2.y);
                    }
                }
                // every lane, every batch: lanes 4r..4r+3 get row (row0 + 64 kb + 8 r)
                const float tot = warp_sum8(rs, lane);
                const int64_t row = row0 + 64 * kb + 8 * (lane >> 2);
                if ((lane & 3) == 0 && row < t.R) D.rowpart[t.rowpart_off + (b * t.R + row) * t.ncb + it.cb] = tot;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                cacc[2 * q] = c2[q].x;
                cacc[2 * q + 1] = c2[q].y;
            }
        } else {
            for (int kk = 0; kk < kTR / 8; ++kk) {
                const int64_t row = row0 + 8 * kk;
                if (row >= t.R) break;   // same for the whole warp
                uint32_t v[8];
                load8(g + (b * t.R + row) * t.C + col0, ncols, v);
                float rs = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < ncols) {
                        const float q = qval(bf16_to_f32(v[j]), k);
                        rs = __fadd_rn(rs, q);
                        cacc[j] = __fadd_rn(cacc[j], q);
                    }
                }
                rs = warp_sum_f32(rs);
                if (lane == 0) D.rowpart[t.rowpart_off + (b * t.R + row) * t.ncb + it.cb] = rs;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) cols[warp][lane * 8 + j] = cacc[j];
        __syncthreads();
        const int c = threadIdx.x;
        const float s = __fadd_rn(__fadd_rn(__fadd_rn(cols[0][c], cols[1][c]), __fadd_rn(cols[2][c], cols[3][c])),
                                  __fadd_rn(__fadd_rn(cols[4][c], cols[5][c]), __fadd_rn(cols[6][c], cols[7][c])));
        const int64_t col = (int64_t)it.cb * kTC + c;
        if (col < t.C) D.colpart[t.colpart_off + (b * t.nbands + it.band) * t.C + col] = s;
        return;
    }

    float acc = 0.f;
    if (it.cls == kTiny) {
        // kTinyPerCta matrices in sub-batches (one matrix per thread), gradients and statistics
        // staged through shared memory; when every sub-batch is whole and aligned, the next
        // sub-batch's copies are in flight while the current one is computed
        const int r = (int)t.R, c = (int)t.C, rc = r * c, sub = tiny_sub(r, c);
        // buffer b: words at smem + b*kTinyWords*2, statistics after both word buffers
        auto words = [&](int b) { return reinterpret_cast<uint16_t*>(smem + b * (kTinyWords * 2)); };
        auto stats = [&](int b) { return reinterpret_cast<float*>(smem + 2 * kTinyWords * 2 + b * (kTinyStats * 4)); };
        const int64_t mend = t.B < (int64_t)it.x + kTinyPerCta ? t.B : (int64_t)it.x + kTinyPerCta;
        const int64_t nmat = mend - it.x;
        const bool pipe = nmat % sub == 0 && aligned16(g) && aligned16(t.row) && aligned16(t.col);
        const int nsub = (int)((nmat + sub - 1) / sub);
        if (pipe && r == 3 && c == 3) {
            acc = kP ? conv3_stats<true>(g, t.row, t.col, it.x, nsub, smem, k)
                              : conv3_stats<false>(g, t.row, t.col, it.x, nsub, smem, k);
        } else if (pipe) {
            for (int kk = -1; kk < nsub; ++kk) {
                // issue sub-batch kk+1 (its buffer was released by the barrier ending kk-1)
                if (kk + 1 < nsub) {
                    const int64_t m1 = it.x + (int64_t)(kk + 1) * sub;
                    const int b1 = (kk + 1) & 1;
                    stage_async(words(b1), g + m1 * rc, sub * rc * 2);
                    stage_async(stats(b1), t.row + m1 * r, sub * r * 4);
                    stage_async(stats(b1) + sub * r, t.col + m1 * c, sub * c * 4);
                    cp_async_commit();
                }
                if (kk < 0) continue;
                if (kk + 1 < nsub) cp_async_wait<1>();
                else cp_async_wait<0>();
                __syncthreads();
                const int b = kk & 1, i = threadIdx.x;
                float* sR = stats(b);
                float* sC = sR + sub * r;
                if (i < sub) {
                    const uint16_t* gm = words(b) + i * rc;
                    float a;
                    if (r == 3 && c == 3)
                        a = kP ? stats3<true>(gm, sR + i * r, sC + i * c, k) : stats3<false>(gm, sR + i * r, sC + i * c, k);
                    else
                        a = tiny_stats_any(gm, sR + i * r, sC + i * c, r, c, k);
                    acc = __fadd_rn(acc, a);
                }
                __syncthreads();
                const int64_t m0 = it.x + (int64_t)kk * sub;
                unstage(t.row + m0 * r, sR, sub * r, false);
                unstage(t.col + m0 * c, sC, sub * c, false);
                __syncthreads();
            }
        } else {
            for (int kk = 0; kk < nsub; ++kk) {
                const int64_t m0 = it.x + (int64_t)kk * sub;
                const int nm = (int)(mend - m0 < sub ? mend - m0 : sub);
                float* sR = stats(0);
                float* sC = sR + nm * r;
                stage(words(0), g + m0 * rc, nm * rc);
                stage(sR, t.row + m0 * r, nm * r);
                stage(sC, t.col + m0 * c, nm * c);
                __syncthreads();
                const int i = threadIdx.x;
                if (i < nm) {
                    const uint16_t* gm = words(0) + i * rc;
                    acc = __fadd_rn(acc, tiny_stats_call(gm, sR + i * r, sC + i * c, r, c, k));
                }
                __syncthreads();
                unstage(t.row + m0 * r, sR, nm * r, false);
                unstage(t.col + m0 * c, sC, nm * c, false);
                __syncthreads();
            }
        }
    } else {  // kVec
        const int64_t e0 = (int64_t)it.x * kVecPerCta;
        const int64_t e1 = (t.numel < e0 + kVecPerCta ? t.numel : e0 + kVecPerCta);
        for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
            const float gg = bf16_to_f32(g[e]);
            const float nv = ema(t.col[e], qval(gg, k), k);
            t.col[e] = nv;
            const float u = numer<kP>(__fmul_rn(rsqrt_rn(nv), gg), k);
            acc = __fadd_rn(acc, __fmul_rn(u, u));
        }
    }
    const float tot = block_sum(acc, sm);
    finish_ss(D, t, it.tensor, it.part, tot, k, sm);
}

// ------------------------------------------------------------------------------------ finalize
__global__ void __launch_bounds__(kThreads) k_final(Dev D, const Item* items, K k) {
    __shared__ float sm[32];
    __shared__ float part[kFinGroups][kFinColsPerItem];
    __shared__ bool last;
    const Item it = items[blockIdx.x];
    const FTensor t = D.tensors[it.tensor];
    const int64_t b = it.x;
    pdl_sync();
    load_k(k);
    if (it.cls == kFinRows) {
        // R EMA of 256 rows (one per thread), their sum, and mean(R) by the matrix's last block
        const int64_t i = (int64_t)it.cb * kFinRowsPerItem + threadIdx.x;
        float nr = 0.f;
        if (i < t.R) {
            const float* rp = D.rowpart + t.rowpart_off + (b * t.R + i) * t.ncb;
            Comp s;
            int cb = 0;
            for (; cb + 4 <= t.ncb; cb += 4) {   // four independent loads in flight
                const float x0 = rp[cb], x1 = rp[cb + 1], x2 = rp[cb + 2], x3 = rp[cb + 3];
                s.add(x0);
                s.add(x1);
                s.add(x2);
                s.add(x3);
            }
            for (; cb < t.ncb; ++cb) s.add(rp[cb]);
            nr = ema(t.row[b * t.R + i], __fdiv_rn(s.value(), (float)t.C), k);
            t.row[b * t.R + i] = nr;
        }
        const float tot = block_sum(nr, sm);
        const int64_t mat = t.mat_off + b;
        if (threadIdx.x == 0) {
            D.rbarpart[t.rbarpart_off + b * t.n_rowitems + it.cb] = tot;
            __threadfence();
            last = atomicAdd(&D.rcounter[mat], 1u) == (unsigned)t.n_rowitems - 1u;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
        Comp acc;
        for (int r = threadIdx.x; r < t.n_rowitems; r += kThreads)
            acc.add(__ldcg(D.rbarpart + t.rbarpart_off + b * t.n_rowitems + r));
        const float all = block_sum(acc.value(), sm);
        if (threadIdx.x == 0) {
            D.rbar[mat] = __fdiv_rn(all, (float)t.R);
            D.rcounter[mat] = 0u;
        }
    } else {
        // C EMA of 32 columns: 8 warps split the row bands (band = warp + 8*n), combined in order
        const int cl = threadIdx.x & (kFinColsPerItem - 1), grp = threadIdx.x / kFinColsPerItem;
        const int64_t j = (int64_t)it.cb * kFinColsPerItem + cl;
        Comp s;
        if (j < t.C) {
            const float* cp = D.colpart + t.colpart_off + b * t.nbands * t.C + j;
            int band = grp;
            for (; band + 3 * kFinGroups < t.nbands; band += 4 * kFinGroups) {   // four loads in flight
                const float x0 = cp[(int64_t)band * t.C], x1 = cp[(int64_t)(band + kFinGroups) * t.C];
                const float x2 = cp[(int64_t)(band + 2 * kFinGroups) * t.C], x3 = cp[(int64_t)(band + 3 * kFinGroups) * t.C];
                s.add(x0);
                s.add(x1);
                s.add(x2);
                s.add(x3);
            }
            for (; band < t.nbands; band += kFinGroups) s.add(cp[(int64_t)band * t.C]);
        }
        part[grp][cl] = s.value();
        __syncthreads();
        if (grp == 0 && j < t.C) {
            const float c = __fadd_rn(__fadd_rn(__fadd_rn(part[0][cl], part[1][cl]), __fadd_rn(part[2][cl], part[3][cl])),
                                      __fadd_rn(__fadd_rn(part[4][cl], part[5][cl]), __fadd_rn(part[6][cl], part[7][cl])));
            const float nc = ema(t.col[b * t.C + j], __fdiv_rn(c, (float)t.R), k);
            t.col[b * t.C + j] = nc;
            D.cc[t.cc_off + b * t.C + j] = rsqrt_rn(nc);
        }
    }
}

// ------------------------------------------------------------------------------------ rms
template <bool kP>
__global__ void __launch_bounds__(kThreads, 4) k_rms(Dev D, const Item* items, K k) {
    __shared__ float sm[32];
    const Item it = items[blockIdx.x];
    const FTensor t = D.tensors[it.tensor];
    const uint16_t* __restrict__ g = D.grads[it.tensor];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = it.x;
    const int64_t col0 = (int64_t)it.cb * kTC + lane * 8;
    const int ncols = cols_in(t.C - col0);
    const bool vec = aligned16(g) && (t.C % 8 == 0);      // same for every lane of the block
    const bool lane_ok = ncols == 8;                       // C % 8 == 0: 8 or 0 columns
    const int64_t row0 = (int64_t)it.band * kTR + warp;
    // the first eight rows' gradients are loaded before waiting for the finalize kernel
    const uint64_t keep = l2_keep_policy();
    uint4 x[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int64_t row = row0 + 8 * kk;
        x[kk] = (vec && row < t.R && lane_ok)
                    ? ld_keep(reinterpret_cast<const uint4*>(g + (b * t.R + row) * t.C + col0), keep) : make_uint4(0, 0, 0, 0);
    }
    pdl_sync();
    load_k(k);
    const float rbar = D.rbar[t.mat_off + b];
    float ccv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ccv[j] = j < ncols ? D.cc[t.cc_off + b * t.C + col0 + j] : 0.f;
    float acc = 0.f;
    if (vec) {
        // row factor rsqrt(R_i / mean R) of the warp's 16 rows: lane l (and l + 16) computes row
        // row0 + 8 l, each row's value is then broadcast by one shuffle
        const int64_t my_row = row0 + 8 * (lane & 15);
        const float rr_mine = my_row < t.R ? rsqrt_rn(__fdiv_rn(t.row[b * t.R + my_row], rbar)) : 0.f;
        const float2 cc2[4] = {make_float2(ccv[0], ccv[1]), make_float2(ccv[2], ccv[3]), make_float2(ccv[4], ccv[5]),
                               make_float2(ccv[6], ccv[7])};
        float2 acc2 = f2(0.f);
        constexpr bool prodigy = kP;
        const float2 un2 = f2(k.unum);
#pragma unroll 1
        for (int kb = 0; kb < kTR / 64; ++kb) {
            if (kb > 0) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int64_t row = row0 + 64 * kb + 8 * kk;
                    x[kk] = (row < t.R && lane_ok)
                                ? ld_keep(reinterpret_cast<const uint4*>(g + (b * t.R + row) * t.C + col0), keep) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int64_t row = row0 + 64 * kb + 8 * kk;
                const float rr = __shfl_sync(0xFFFFFFFFu, rr_mine, 8 * kb + kk);   // every lane
                if (lane_ok && row < t.R) {
                    const uint32_t wd[4] = {x[kk].x, x[kk].y, x[kk].z, x[kk].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float2 u = __fmul2_rn(__fmul2_rn(f2(rr), cc2[q]), bf16x2_to_f2(wd[q]));
                        if (prodigy) u = __fmul2_rn(u, un2);
                        acc2 = __ffma2_rn(u, u, acc2);
                    }
                }
            }
        }
        acc = __fadd_rn(acc2.x, acc2.y);
    } else {
        for (int kk = 0; kk < kTR / 8; ++kk) {
            const int64_t row = row0 + 8 * kk;
            if (row >= t.R) break;
            const float rr = rsqrt_rn(__fdiv_rn(t.row[b * t.R + row], rbar));
            uint32_t v[8];
            load8(g + (b * t.R + row) * t.C + col0, ncols, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j < ncols) {
                    const float u = numer<kP>(__fmul_rn(__fmul_rn(rr, ccv[j]), bf16_to_f32(v[j])), k);
                    acc = __fadd_rn(acc, __fmul_rn(u, u));
                }
            }
        }
    }
    const float tot = block_sum(acc, sm);
    finish_ss(D, t, it.tensor, it.part, tot, k, sm);
}

// ------------------------------------------------------------------------------------ apply
// Applies the update to the eight elements of one row held in (Wv, Rv) with gradients G, in
// packed pairs: u = (rr * cc_j) * g_j (times d in Prodigy mode);  w = w + w*nwdlr (when decaying);
// w = w + u*(-s);  split.
__device__ __forceinline__ void apply8x2(const uint4& G, uint4& Wv, uint4& Rv, float rr, const float2 (&cc2)[4],
                                         bool has_res, bool decay, float2 nwd2, float2 ns2, bool prodigy, float2 un2) {
    const uint32_t g32[4] = {G.x, G.y, G.z, G.w};
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&Wv);
    uint32_t* r32 = reinterpret_cast<uint32_t*>(&Rv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float2 w2 = has_res ? make_float2(__uint_as_float(__byte_perm(r32[q], w32[q], 0x5410)),
                                          __uint_as_float(__byte_perm(r32[q], w32[q], 0x7632)))
                            : bf16x2_to_f2(w32[q]);
        float2 u2 = __fmul2_rn(__fmul2_rn(f2(rr), cc2[q]), bf16x2_to_f2(g32[q]));
        if (prodigy) u2 = __fmul2_rn(u2, un2);
        if (decay) w2 = __fadd2_rn(w2, __fmul2_rn(w2, nwd2));
        w2 = __fadd2_rn(w2, __fmul2_rn(u2, ns2));
        const uint32_t b0 = __float_as_uint(w2.x), b1 = __float_as_uint(w2.y);
        if (has_res) {
            w32[q] = pack_hi16(b0, b1);
            r32[q] = pack_lo16(b0, b1);
        } else {
            w32[q] = pack_lo16(rne_bf16(w2.x), rne_bf16(w2.y));
        }
    }
}

template <bool kP>
__global__ void __launch_bounds__(kThreads, 4) k_apply(Dev D, const Item* items, K k) {
    __shared__ __align__(16) unsigned char smem[kApplySmem];
    const Item it = items[blockIdx.x];
    const FTensor t = D.tensors[it.tensor];
    const uint16_t* __restrict__ g = D.grads[it.tensor];
    const bool has_res = t.res != nullptr;
    uint32_t nf = 0u;   // largest bf16 magnitude this thread stored (non-finite detection)

    if (it.cls == kWide) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int64_t b = it.x;
        const int64_t col0 = (int64_t)it.cb * kTC + lane * 8;
        const int ncols = cols_in(t.C - col0);
        const bool vec = aligned16(g) && aligned16(t.w) && (!has_res || aligned16(t.res)) && (t.C % 8 == 0);
        const int64_t row0 = (int64_t)it.band * kTR + warp;
        if (vec) {
            const bool lane_ok = ncols == 8;   // C % 8 == 0: a lane's group is whole or empty
            // two rows per iteration, all six 128-bit loads issued before the arithmetic; the
            // first pair is loaded before waiting for the RMS kernel (gradients and weights are
            // written by no earlier kernel of the step)
            uint4 GA = make_uint4(0, 0, 0, 0), WA = GA, RA = GA, GB = GA, WB = GA, RB = GA;
            auto load_pair = [&](int kk) {
                const int64_t rowA = row0 + 8 * kk;
                if (rowA >= t.R || !lane_ok) return;
                const int64_t offA = (b * t.R + rowA) * t.C + col0, offB = offA + 8 * t.C;
                GA = __ldcg(reinterpret_cast<const uint4*>(g + offA));
                WA = ld_stream(reinterpret_cast<const uint4*>(t.w + offA));
                if (has_res) RA = ld_stream(reinterpret_cast<const uint4*>(t.res + offA));
                if (rowA + 8 < t.R) {
                    GB = __ldcg(reinterpret_cast<const uint4*>(g + offB));
                    WB = ld_stream(reinterpret_cast<const uint4*>(t.w + offB));
                    if (has_res) RB = ld_stream(reinterpret_cast<const uint4*>(t.res + offB));
                }
            };
            load_pair(0);
            pdl_sync();
            load_k(k);
            const float us = update_scale(D.den[it.tensor], k);
            const float2 ns2 = f2(-us), nwd2 = f2(k.nwdlr), un2 = f2(k.unum);
            const bool decay = k.nwdlr != 0.0f;
            constexpr bool prodigy = kP;
            float2 cc2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                cc2[q] = lane_ok ? make_float2(D.cc[t.cc_off + b * t.C + col0 + 2 * q], D.cc[t.cc_off + b * t.C + col0 + 2 * q + 1])
                                 : f2(0.f);
            const float rbar = D.rbar[t.mat_off + b];
            // row factors of the warp's 16 rows, one per lane (l and l + 16), broadcast per row
            const int64_t my_row = row0 + 8 * (lane & 15);
            const float rr_mine = my_row < t.R ? rsqrt_rn(__fdiv_rn(t.row[b * t.R + my_row], rbar)) : 0.f;
#pragma unroll 1
            for (int kk = 0; kk < kTR / 8; kk += 2) {
                const int64_t rowA = row0 + 8 * kk, rowB = rowA + 8;
                if (rowA >= t.R) break;   // the same for every lane of the warp
                const float rrA = __shfl_sync(0xFFFFFFFFu, rr_mine, kk);
                const float rrB = __shfl_sync(0xFFFFFFFFu, rr_mine, kk + 1);
                if (!lane_ok) continue;
                const bool hasB = rowB < t.R;
                const int64_t offA = (b * t.R + rowA) * t.C + col0, offB = offA + 8 * t.C;
                if (kk > 0) load_pair(kk);
                apply8x2(GA, WA, RA, rrA, cc2, has_res, decay, nwd2, ns2, prodigy, un2);
                nf = max_bf16_mag(nf, WA);
                st_stream(reinterpret_cast<uint4*>(t.w + offA), WA);
                if (has_res) st_stream(reinterpret_cast<uint4*>(t.res + offA), RA);
                if (hasB) {
                    apply8x2(GB, WB, RB, rrB, cc2, has_res, decay, nwd2, ns2, prodigy, un2);
                    nf = max_bf16_mag(nf, WB);
                    st_stream(reinterpret_cast<uint4*>(t.w + offB), WB);
                    if (has_res) st_stream(reinterpret_cast<uint4*>(t.res + offB), RB);
                }
            }
        } else {
            pdl_sync();
            load_k(k);
            const float us = update_scale(D.den[it.tensor], k);
            float ccv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) ccv[j] = j < ncols ? D.cc[t.cc_off + b * t.C + col0 + j] : 0.f;
            const float rbar = D.rbar[t.mat_off + b];
            for (int kk = 0; kk < kTR / 8; ++kk) {
                const int64_t row = row0 + 8 * kk;
                if (row >= t.R) break;
                const float rr = rsqrt_rn(__fdiv_rn(t.row[b * t.R + row], rbar));
                const int64_t off = (b * t.R + row) * t.C + col0;
                for (int j = 0; j < ncols; ++j) {
                    uint32_t hi = t.w[off + j], lo = has_res ? t.res[off + j] : 0u;
                    const float u = numer<kP>(__fmul_rn(__fmul_rn(rr, ccv[j]), bf16_to_f32(g[off + j])), k);
                    apply_elem(hi, lo, has_res, u, us, k);
                    nf = max(nf, hi & 0x7FFFu);
                    t.w[off + j] = (uint16_t)hi;
                    if (has_res) t.res[off + j] = (uint16_t)lo;
                }
            }
        }
        count_nonfinite(D, nf);
        return;
    }
    pdl_sync();
    load_k(k);
    const float us = update_scale(D.den[it.tensor], k);
    if (it.cls == kTiny) {
        // as in k_stats: sub-batches staged through shared memory, double-buffered when whole
        // and aligned; w and res are updated in shared memory and streamed back
        const int r = (int)t.R, c = (int)t.C, rc = r * c, sub = tiny_sub(r, c);
        constexpr int kBuf = 3 * kTinyWords * 2 + kTinyStats * 4;
        uint16_t* sg[2];
        uint16_t* sw[2];
        uint16_t* sr[2];
        float* sf[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            sg[b] = reinterpret_cast<uint16_t*>(smem + b * kBuf);
            sw[b] = sg[b] + kTinyWords;
            sr[b] = sw[b] + kTinyWords;
            sf[b] = reinterpret_cast<float*>(sr[b] + kTinyWords);
        }
        const int64_t mend = t.B < (int64_t)it.x + kTinyPerCta ? t.B : (int64_t)it.x + kTinyPerCta;
        const int64_t nmat = mend - it.x;
        const bool pipe = nmat % sub == 0 && aligned16(g) && aligned16(t.w) && (!has_res || aligned16(t.res)) &&
                          aligned16(t.row) && aligned16(t.col);
        const int nsub = (int)((nmat + sub - 1) / sub);
        if (pipe && r == 3 && c == 3) {
            const float un = k.unum, nw = k.nwdlr;
            if (has_res) {
                if (nw != 0.0f) nf = conv3_apply<true, true, kP>(g, t.w, t.res, t.row, t.col, it.x, nsub, smem, us, nw, un);
                else nf = conv3_apply<true, false, kP>(g, t.w, t.res, t.row, t.col, it.x, nsub, smem, us, nw, un);
            } else {
                if (nw != 0.0f) nf = conv3_apply<false, true, kP>(g, t.w, t.res, t.row, t.col, it.x, nsub, smem, us, nw, un);
                else nf = conv3_apply<false, false, kP>(g, t.w, t.res, t.row, t.col, it.x, nsub, smem, us, nw, un);
            }
            count_nonfinite(D, nf);
            return;
        }
        auto compute = [&](int b, int nm) {
            const int i = threadIdx.x;
            if (i >= nm) return;
            const float* sR = sf[b];
            const float* sC = sf[b] + nm * r;
            if (r == 3 && c == 3) {
                uint16_t* wm = sw[b] + i * rc;
                uint16_t* rm = sr[b] + i * rc;
                const uint16_t* gm = sg[b] + i * rc;
                const float* Rs = sR + i * r;
                const float* Cs = sC + i * c;
                if (has_res) {
                    if (k.nwdlr != 0.0f) apply3<true, true, kP>(wm, rm, gm, Rs, Cs, us, k.nwdlr, k.unum);
                    else apply3<true, false, kP>(wm, rm, gm, Rs, Cs, us, k.nwdlr, k.unum);
                } else {
                    if (k.nwdlr != 0.0f) apply3<false, true, kP>(wm, rm, gm, Rs, Cs, us, k.nwdlr, k.unum);
                    else apply3<false, false, kP>(wm, rm, gm, Rs, Cs, us, k.nwdlr, k.unum);
                }
            } else
                tiny_apply_any<kP>(sw[b] + i * rc, sr[b] + i * rc, sg[b] + i * rc, sR + i * r, sC + i * c, r, c, has_res, us, k);
            for (int e = 0; e < rc; ++e) nf = max(nf, (uint32_t)(sw[b][i * rc + e] & 0x7FFFu));
        };
        if (pipe) {
            auto issue = [&](int kk) {
                const int64_t m0 = it.x + (int64_t)kk * sub;
                const int b = kk & 1;
                stage_async(sg[b], g + m0 * rc, sub * rc * 2);
                stage_async(sw[b], t.w + m0 * rc, sub * rc * 2);
                if (has_res) stage_async(sr[b], t.res + m0 * rc, sub * rc * 2);
                stage_async(sf[b], t.row + m0 * r, sub * r * 4);
                stage_async(sf[b] + sub * r, t.col + m0 * c, sub * c * 4);
                cp_async_commit();
            };
            issue(0);
            for (int kk = 0; kk < nsub; ++kk) {
                if (kk + 1 < nsub) {
                    issue(kk + 1);   // its buffer was released by the barrier ending iteration kk-1
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncthreads();
                const int b = kk & 1;
                compute(b, sub);
                __syncthreads();
                const int64_t m0 = it.x + (int64_t)kk * sub;
                unstage(t.w + m0 * rc, sw[b], sub * rc, true);
                if (has_res) unstage(t.res + m0 * rc, sr[b], sub * rc, true);
                __syncthreads();
            }
        } else {
            for (int kk = 0; kk < nsub; ++kk) {
                const int64_t m0 = it.x + (int64_t)kk * sub;
                const int nm = (int)(mend - m0 < sub ? mend - m0 : sub);
                stage(sg[0], g + m0 * rc, nm * rc);
                stage(sw[0], t.w + m0 * rc, nm * rc);
                if (has_res) stage(sr[0], t.res + m0 * rc, nm * rc);
                stage(sf[0], t.row + m0 * r, nm * r);
                stage(sf[0] + nm * r, t.col + m0 * c, nm * c);
                __syncthreads();
                compute(0, nm);
                __syncthreads();
                unstage(t.w + m0 * rc, sw[0], nm * rc, true);
                if (has_res) unstage(t.res + m0 * rc, sr[0], nm * rc, true);
                __syncthreads();
            }
        }
        count_nonfinite(D, nf);
        return;
    }
    const int64_t e0 = (int64_t)it.x * kVecPerCta;
    const int64_t e1 = (t.numel < e0 + kVecPerCta ? t.numel : e0 + kVecPerCta);
    for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
        uint32_t hi = t.w[e], lo = has_res ? t.res[e] : 0u;
        const float u = numer<kP>(__fmul_rn(rsqrt_rn(t.col[e]), bf16_to_f32(g[e])), k);
        apply_elem(hi, lo, has_res, u, us, k);
        nf = max(nf, hi & 0x7FFFu);
        t.w[e] = (uint16_t)hi;
        if (has_res) t.res[e] = (uint16_t)lo;
    }
    count_nonfinite(D, nf);
}

}  // namespace

// ------------------------------------------------------------------------------------ host plan
struct Wave {
    int32_t item_off, n_wide, n_total;   // items: wide tiles first, then tiny and vector CTAs
    int32_t fin_off, n_fin;
};

struct FactoredPlan {
    Dev dev{};
    FTensor* d_tensors = nullptr;
    Item* d_items = nullptr;
    Item* d_fin = nullptr;
    std::vector<Wave> waves;
    std::vector<void*> allocs;
    // waves are independent (disjoint tensors and scratch), so consecutive waves run on
    // different streams: the caller's and n_aux internal ones, forked from and joined back into
    // the caller's stream by events
    int n_aux = 0;
    cudaStream_t aux[kWaveStreams > 1 ? kWaveStreams - 1 : 1] = {};
    cudaEvent_t fork_ev = nullptr;
    cudaEvent_t join_ev[kWaveStreams > 1 ? kWaveStreams - 1 : 1] = {};
};

template <class T>
static int alloc_dev(FactoredPlan* p, T** out, size_t count, const char* what) {
    const size_t bytes = std::max<size_t>(count, 1) * sizeof(T);
    if (cudaMalloc(reinterpret_cast<void**>(out), bytes) != cudaSuccess) {
        cudaGetLastError();
        return set_error(OPTIM_ENOMEM, "cudaMalloc(%zu) for %s failed", bytes, what);
    }
    p->allocs.push_back(*out);
    return check_cuda(cudaMemset(*out, 0, bytes), what);
}

// Host-side layout of a factored plan: tensor records, work items and the sizes (in elements)
// of every scratch array.  Shared by the allocating plan below.
struct PlanLayout {
    std::vector<FTensor> ts;
    std::vector<Item> items, fin;
    std::vector<Wave> waves;
    int64_t rowpart = 0, colpart = 0, cc = 0, ss = 0, mats = 0, rbarpart = 0;
};

// Per-tensor classes and scratch offsets (no work items yet).
static void plan_tensors(const std::vector<optim_tensor_desc_t>& desc, PlanLayout& L) {
    const int32_t n = (int32_t)desc.size();
    L.ts.assign(n, FTensor{});
    for (int32_t i = 0; i < n; ++i) {
        const optim_tensor_desc_t& d = desc[i];
        FTensor& t = L.ts[i];
        t.w = static_cast<uint16_t*>(d.w_bf16);
        t.res = static_cast<uint16_t*>(d.res_u16);
        t.numel = d.numel;
        if (d.ndim >= 2) {
            t.R = d.shape[d.ndim - 2];
            t.C = d.shape[d.ndim - 1];
            t.B = 1;
            for (int k = 0; k < d.ndim - 2; ++k) t.B *= d.shape[k];
            t.row = static_cast<float*>(d.m);
            t.col = static_cast<float*>(d.v);
            t.cls = (t.R * t.C <= 16) ? kTiny : kWide;
        } else {
            t.B = 1;
            t.R = 1;
            t.C = d.numel;
            t.col = static_cast<float*>(d.v);
            t.cls = kVec;
        }
        if (d.numel == 0) continue;
        if (t.cls == kWide) {
            t.ncb = (int32_t)((t.C + kTC - 1) / kTC);
            t.nbands = (int32_t)((t.R + kTR - 1) / kTR);
            t.n_rowitems = (int32_t)((t.R + kFinRowsPerItem - 1) / kFinRowsPerItem);
            t.rowpart_off = L.rowpart;
            L.rowpart += t.B * t.R * t.ncb;
            t.colpart_off = L.colpart;
            L.colpart += t.B * t.nbands * t.C;
            t.cc_off = L.cc;
            L.cc += t.B * t.C;
            t.mat_off = L.mats;
            L.mats += t.B;
            t.rbarpart_off = L.rbarpart;
            L.rbarpart += t.B * t.n_rowitems;
            t.ss_cnt = (int32_t)(t.B * t.nbands * t.ncb);
        } else if (t.cls == kTiny) {
            t.ss_cnt = (int32_t)((t.B + kTinyPerCta - 1) / kTinyPerCta);
        } else {
            t.ss_cnt = (int32_t)((t.numel + kVecPerCta - 1) / kVecPerCta);
        }
        t.ss_off = L.ss;
        L.ss += t.ss_cnt;
    }
}

// Work items of one tensor planned by plan_tensors: statistics / RMS / update items, finalize items.
static void item_counts(const FTensor& t, int64_t& items, int64_t& fin) {
    items = fin = 0;
    if (t.numel == 0) return;
    if (t.cls == kWide) {
        items = t.B * t.nbands * t.ncb;
        fin = t.B * (t.n_rowitems + (t.C + kFinColsPerItem - 1) / kFinColsPerItem);
    } else {
        items = t.ss_cnt;
    }
}

// Waves and work items over the tensors planned by plan_tensors.
static void plan_waves(PlanLayout& L) {
    const int32_t n = (int32_t)L.ts.size();
    // waves: consecutive tensors, at most kWaveGradBytes of gradients each (the L2-resident
    // target), balanced so that no wave is much smaller than the others: the group's gradient
    // bytes are split into ceil(total / kWaveGradBytes) near-equal targets
    int64_t total = 0;
    for (int32_t q = 0; q < n; ++q) total += 2 * L.ts[q].numel;
    const int64_t nw = total > 0 ? (total + kWaveGradBytes - 1) / kWaveGradBytes : 1;
    const int64_t target = (total + nw - 1) / nw;
    int32_t i = 0;
    while (i < n) {
        int64_t bytes = 0;
        int32_t j = i;
        while (j < n && (j == i || (bytes + 2 * L.ts[j].numel <= kWaveGradBytes && bytes + L.ts[j].numel <= target)))
            bytes += 2 * L.ts[j++].numel;
        Wave wv{};
        wv.item_off = (int32_t)L.items.size();
        wv.fin_off = (int32_t)L.fin.size();
        for (int32_t q = i; q < j; ++q) {
            const FTensor& t = L.ts[q];
            if (t.numel == 0 || t.cls != kWide) continue;
            int32_t part = 0;
            for (int64_t b = 0; b < t.B; ++b) {
                for (int32_t band = 0; band < t.nbands; ++band)
                    for (int32_t cb = 0; cb < t.ncb; ++cb) L.items.push_back(Item{q, kWide, (int32_t)b, band, cb, part++});
                for (int32_t rb = 0; rb < t.n_rowitems; ++rb) L.fin.push_back(Item{q, kFinRows, (int32_t)b, 0, rb, 0});
                const int32_t ncol = (int32_t)((t.C + kFinColsPerItem - 1) / kFinColsPerItem);
                for (int32_t cb = 0; cb < ncol; ++cb) L.fin.push_back(Item{q, kFinCols, (int32_t)b, 0, cb, 0});
            }
        }
        wv.n_wide = (int32_t)L.items.size() - wv.item_off;
        for (int32_t q = i; q < j; ++q) {
            const FTensor& t = L.ts[q];
            if (t.numel == 0 || t.cls == kWide) continue;
            for (int32_t part = 0; part < t.ss_cnt; ++part) {
                const int32_t x = t.cls == kTiny ? part * kTinyPerCta : part;
                L.items.push_back(Item{q, t.cls, x, 0, 0, part});
            }
        }
        wv.n_total = (int32_t)L.items.size() - wv.item_off;
        wv.n_fin = (int32_t)L.fin.size() - wv.fin_off;
        L.waves.push_back(wv);
        i = j;
    }
}

static void plan_layout(const std::vector<optim_tensor_desc_t>& desc, PlanLayout& L) {
    plan_tensors(desc, L);
    plan_waves(L);
}

int factored_plan_build(FactoredPlan*& plan, const std::vector<optim_tensor_desc_t>& desc) {
    plan = new FactoredPlan();
    FactoredPlan* p = plan;
    PlanLayout L;
    plan_layout(desc, L);
    p->waves = L.waves;
    const size_t n = desc.size();
    int rc = OPTIM_OK;
    Dev& D = p->dev;
    if (!rc) rc = alloc_dev(p, &p->d_tensors, L.ts.size(), "factored tensor table");
    if (!rc) rc = check_cuda(cudaMemcpy(p->d_tensors, L.ts.data(), L.ts.size() * sizeof(FTensor), cudaMemcpyHostToDevice), "upload");
    if (!rc) rc = alloc_dev(p, &p->d_items, L.items.size(), "factored work items");
    if (!rc && !L.items.empty()) rc = check_cuda(cudaMemcpy(p->d_items, L.items.data(), L.items.size() * sizeof(Item), cudaMemcpyHostToDevice), "upload");
    if (!rc) rc = alloc_dev(p, &p->d_fin, L.fin.size(), "factored finalize items");
    if (!rc && !L.fin.empty()) rc = check_cuda(cudaMemcpy(p->d_fin, L.fin.data(), L.fin.size() * sizeof(Item), cudaMemcpyHostToDevice), "upload");
    if (!rc) rc = alloc_dev(p, &D.rowpart, (size_t)L.rowpart, "row partial sums");
    if (!rc) rc = alloc_dev(p, &D.colpart, (size_t)L.colpart, "column partial sums");
    if (!rc) rc = alloc_dev(p, &D.cc, (size_t)L.cc, "column factors");
    if (!rc) rc = alloc_dev(p, &D.rbar, (size_t)L.mats, "row means");
    if (!rc) rc = alloc_dev(p, &D.rbarpart, (size_t)L.rbarpart, "row-mean partials");
    if (!rc) rc = alloc_dev(p, &D.rcounter, (size_t)L.mats, "row-mean counters");
    if (!rc) rc = alloc_dev(p, &D.ss, (size_t)L.ss, "sum-of-squares partials");
    if (!rc) rc = alloc_dev(p, &D.den, n, "clip divisors");
    if (!rc) rc = alloc_dev(p, &D.counter, n, "partial counters");
    D.tensors = p->d_tensors;
    const int n_aux = std::min<int>(kWaveStreams - 1, (int)L.waves.size() - 1);
    if (!rc && n_aux > 0) {
        rc = check_cuda(cudaEventCreateWithFlags(&p->fork_ev, cudaEventDisableTiming), "wave fork event");
        for (int a = 0; !rc && a < n_aux; ++a) {
            rc = check_cuda(cudaStreamCreateWithFlags(&p->aux[a], cudaStreamNonBlocking), "wave stream");
            if (!rc) rc = check_cuda(cudaEventCreateWithFlags(&p->join_ev[a], cudaEventDisableTiming), "wave join event");
            if (!rc) p->n_aux = a + 1;
        }
    }
    return rc;
}

void factored_plan_free(FactoredPlan*& plan) {
    if (!plan) return;
    for (int a = 0; a < (int)(sizeof(plan->aux) / sizeof(plan->aux[0])); ++a) {
        if (plan->aux[a]) cudaStreamDestroy(plan->aux[a]);
        if (plan->join_ev[a]) cudaEventDestroy(plan->join_ev[a]);
    }
    if (plan->fork_ev) cudaEventDestroy(plan->fork_ev);
    for (void* a : plan->allocs) cudaFree(a);
    delete plan;
    plan = nullptr;
}

// Launches one kernel of the step with programmatic stream serialization allowed (the kernel
// may start while its predecessor on the stream drains; it waits with griddepcontrol.wait).
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, int grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

FactoredScalars factored_scalars(const optim_factored_hparams_t* hp, int64_t step, float d) {
    FactoredScalars k{};
    k.mode = hp->mode;
    k.clip = hp->clip_threshold;
    k.eps1 = hp->eps1;
    k.eps2 = hp->eps2;
    if (hp->mode == 0) {
        const double beta2t = 1.0 - std::pow((double)step, (double)hp->decay_rate);
        k.b2t = (float)beta2t;
        k.alpha = (float)(1.0 - beta2t);
        k.lr_eff = hp->lr;
        k.unum = 1.0f;
    } else {
        k.b2t = hp->beta2;
        k.alpha = (float)((double)d * (double)d * (1.0 - (double)hp->beta2));
        k.lr_eff = (float)((double)d * (double)hp->lr);
        k.unum = d;
    }
    k.nwdlr = (float)(-(double)hp->weight_decay * (double)k.lr_eff);
    k.kdev = nullptr;
    return k;
}

int launch_factored_step(const FactoredPlan* p, const uint16_t* const* d_grads, const FactoredScalars& s,
                         cudaStream_t stream, cudaEvent_t mid, unsigned long long* nonfinite, cudaEvent_t apply_wait) {
    K k{s.b2t, s.alpha, s.eps1, s.eps2, s.clip, s.lr_eff, s.nwdlr, s.mode, s.unum, s.kdev};
    const bool kp = s.mode == 1;   // Prodigy mode: kernels that apply the numerator factor d
    Dev D = p->dev;
    D.grads = d_grads;
    D.nonfinite = nonfinite;
    const int ns = 1 + p->n_aux;   // streams in use: wave w runs on stream w % ns (0 = caller's)
    int rc = OPTIM_OK;
    if (ns > 1) {
        rc = check_cuda(cudaEventRecord(p->fork_ev, stream), "wave fork");
        for (int a = 0; !rc && a < p->n_aux; ++a) rc = check_cuda(cudaStreamWaitEvent(p->aux[a], p->fork_ev, 0), "wave fork");
        if (rc) return rc;
    }
    for (size_t w = 0; w < p->waves.size() && !rc; ++w) {
        const Wave& wv = p->waves[w];
        const cudaStream_t st = (w % ns == 0) ? stream : p->aux[w % ns - 1];
        const Item* items = p->d_items + wv.item_off;
        const Item* fin = p->d_fin + wv.fin_off;
        if (wv.n_total > 0) rc = check_cuda((kp ? launch_pdl(k_stats<true>, wv.n_total, st, D, items, k)
                                                  : launch_pdl(k_stats<false>, wv.n_total, st, D, items, k)), "factored stats launch");
        if (!rc && wv.n_fin > 0) rc = check_cuda(launch_pdl(k_final, wv.n_fin, st, D, fin, k), "factored finalize launch");
        if (!rc && wv.n_wide > 0) rc = check_cuda((kp ? launch_pdl(k_rms<true>, wv.n_wide, st, D, items, k)
                                                            : launch_pdl(k_rms<false>, wv.n_wide, st, D, items, k)), "factored rms launch");
        if (!rc && mid && w + 1 == p->waves.size()) rc = check_cuda(cudaEventRecord(mid, st), "profile event");
        // the first update on each stream waits for apply_wait; later ones follow it on the stream
        if (!rc && apply_wait && (int)w < ns) rc = check_cuda(cudaStreamWaitEvent(st, apply_wait, 0), "apply wait");
        if (!rc && wv.n_total > 0) rc = check_cuda((kp ? launch_pdl(k_apply<true>, wv.n_total, st, D, items, k)
                                                              : launch_pdl(k_apply<false>, wv.n_total, st, D, items, k)), "factored apply launch");
    }
    // join every internal stream back into the caller's (also after a launch error, so that no
    // internal stream is left ahead of the caller's)
    for (int a = 0; a < p->n_aux && ns > 1; ++a) {
        int r2 = check_cuda(cudaEventRecord(p->join_ev[a], p->aux[a]), "wave join");
        if (!r2) r2 = check_cuda(cudaStreamWaitEvent(stream, p->join_ev[a], 0), "wave join");
        if (!rc) rc = r2;
    }
    return rc;
}

}  // namespace lmo
// ------------------------------------------------------------------------------------ no-alloc
// A single-tensor factored step for callers that cannot allocate device memory: all of its
// scratch (tensor record, work items, gradient-pointer slot, partial sums, column factors, row
// means, sum-of-squares partials, clip divisor, counters) lives in one fixed file-scope device
// array.  The array is created with the module on every GPU that loads the library and stays
// until the process exits; all calls share it.
namespace lmo {
namespace {

constexpr size_t kNoAllocScratchBytes = 32ull << 20;   // 32 MiB per device
constexpr int kNoAllocMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device (host
// code cannot use the symbol itself: its host-side name is only a stand-in).
int noalloc_scratch(void** out) {
    int dev = 0;
    int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(OPTIM_EINVAL, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        rc = check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(no-alloc scratch)");
        if (rc) return rc;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return OPTIM_OK;
}

size_t carve(size_t& off, size_t bytes) {
    const size_t at = off;
    off = (off + bytes + 255) & ~size_t(255);
    return at;
}

}  // namespace
}  // namespace lmo

extern "C" int optim_step_factored_noalloc(const optim_tensor_desc_t* tensor, const void* grad_bf16, int64_t step,
                                           const optim_factored_hparams_t* hp, void* stream) {
    using namespace lmo;
    if (!tensor || !hp) return set_error(OPTIM_EINVAL, "tensor or hparams is NULL");
    const optim_tensor_desc_t& d = *tensor;
    if (step < 1) return set_error(OPTIM_EINVAL, "step %lld < 1", (long long)step);
    if (d.numel < 0 || d.ndim < 1 || d.ndim > 4) return set_error(OPTIM_EINVAL, "bad numel or ndim");
    int64_t prod = 1;
    for (int k = 0; k < d.ndim; ++k) {
        if (d.shape[k] < 0) return set_error(OPTIM_EINVAL, "negative dim");
        prod *= d.shape[k];
    }
    if (prod != d.numel) return set_error(OPTIM_EINVAL, "shape product %lld != numel %lld", (long long)prod, (long long)d.numel);
    if (d.numel == 0) return OPTIM_OK;
    if (!d.w_bf16 || !d.v || (d.ndim >= 2 && !d.m) || !grad_bf16)
        return set_error(OPTIM_EINVAL, "weight, state or gradient pointer is NULL");
    if (!is_aligned(d.w_bf16, 2) || (d.res_u16 && !is_aligned(d.res_u16, 2)) || !is_aligned(grad_bf16, 2) ||
        !is_aligned(d.v, 4) || (d.m && !is_aligned(d.m, 4)))
        return set_error(OPTIM_EALIGN, "a buffer is not aligned to its element size");
    // the same checks as optim_step_factored (finite, non-negative lr, decay, eps1, eps2, d)
    auto finite_nonneg = [](float x) { return std::isfinite(x) && x >= 0.0f; };
    if (!finite_nonneg(hp->lr) || !(hp->clip_threshold > 0.0f) || !std::isfinite(hp->clip_threshold) ||
        !finite_nonneg(hp->weight_decay) || !finite_nonneg(hp->eps1) || !finite_nonneg(hp->eps2) ||
        (hp->mode != 0 && hp->mode != 1) || !std::isfinite(hp->decay_rate) ||
        (hp->mode == 1 && (!(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) || !finite_nonneg(hp->d))))
        return set_error(OPTIM_EINVAL, "invalid factored hyper-parameters");

    // layout of this tensor's plan inside the fixed scratch, sized from the tensor's shape before
    // any work item is built (an oversized tensor is rejected without building its tables)
    PlanLayout L;
    plan_tensors(std::vector<optim_tensor_desc_t>(1, d), L);
    int64_t n_items = 0, n_fin = 0;
    item_counts(L.ts[0], n_items, n_fin);
    size_t off = 0;
    const size_t o_ts = carve(off, sizeof(FTensor));
    const size_t o_items = carve(off, (size_t)n_items * sizeof(Item));
    const size_t o_fin = carve(off, (size_t)n_fin * sizeof(Item));
    const size_t o_grad = carve(off, sizeof(void*));
    const size_t o_rowpart = carve(off, (size_t)L.rowpart * 4), o_colpart = carve(off, (size_t)L.colpart * 4);
    const size_t o_cc = carve(off, (size_t)L.cc * 4), o_rbar = carve(off, (size_t)L.mats * 4);
    const size_t o_rbarpart = carve(off, (size_t)L.rbarpart * 4), o_rcounter = carve(off, (size_t)L.mats * 4);
    const size_t o_ss = carve(off, (size_t)L.ss * 4), o_den = carve(off, 4), o_counter = carve(off, 4);
    if (off > kNoAllocScratchBytes)
        return set_error(OPTIM_EINVAL, "tensor of %lld elements needs %zu bytes of scratch; the fixed no-alloc scratch holds %zu",
                         (long long)d.numel, off, kNoAllocScratchBytes);
    plan_waves(L);
    if ((int64_t)L.items.size() != n_items || (int64_t)L.fin.size() != n_fin)
        return set_error(OPTIM_EINVAL, "internal: work-item count differs from its estimate");

    void* base = nullptr;
    int rc = noalloc_scratch(&base);
    if (rc) return rc;
    char* sb = static_cast<char*>(base);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const FactoredScalars k = factored_scalars(hp, step, hp->d);

    // tables (pageable host memory: staged by the runtime before the call returns), counters
    // cleared because the previous call's contents stay in the shared array
    const void* gp = grad_bf16;
    rc = check_cuda(cudaMemcpyAsync(sb + o_ts, L.ts.data(), sizeof(FTensor), cudaMemcpyHostToDevice, s), "no-alloc upload");
    if (!rc && !L.items.empty())
        rc = check_cuda(cudaMemcpyAsync(sb + o_items, L.items.data(), L.items.size() * sizeof(Item), cudaMemcpyHostToDevice, s), "no-alloc upload");
    if (!rc && !L.fin.empty())
        rc = check_cuda(cudaMemcpyAsync(sb + o_fin, L.fin.data(), L.fin.size() * sizeof(Item), cudaMemcpyHostToDevice, s), "no-alloc upload");
    if (!rc) rc = check_cuda(cudaMemcpyAsync(sb + o_grad, &gp, sizeof(void*), cudaMemcpyHostToDevice, s), "no-alloc upload");
    if (!rc && L.mats) rc = check_cuda(cudaMemsetAsync(sb + o_rcounter, 0, (size_t)L.mats * 4, s), "no-alloc clear");
    if (!rc) rc = check_cuda(cudaMemsetAsync(sb + o_counter, 0, 4, s), "no-alloc clear");
    if (rc) return rc;

    FactoredPlan plan;
    plan.waves = L.waves;
    plan.d_tensors = reinterpret_cast<FTensor*>(sb + o_ts);
    plan.d_items = reinterpret_cast<Item*>(sb + o_items);
    plan.d_fin = reinterpret_cast<Item*>(sb + o_fin);
    Dev& D = plan.dev;
    D.tensors = plan.d_tensors;
    D.rowpart = reinterpret_cast<float*>(sb + o_rowpart);
    D.colpart = reinterpret_cast<float*>(sb + o_colpart);
    D.cc = reinterpret_cast<float*>(sb + o_cc);
    D.rbar = reinterpret_cast<float*>(sb + o_rbar);
    D.rbarpart = reinterpret_cast<float*>(sb + o_rbarpart);
    D.rcounter = reinterpret_cast<unsigned*>(sb + o_rcounter);
    D.ss = reinterpret_cast<float*>(sb + o_ss);
    D.den = reinterpret_cast<float*>(sb + o_den);
    D.counter = reinterpret_cast<unsigned*>(sb + o_counter);
    return launch_factored_step(&plan, reinterpret_cast<const uint16_t* const*>(sb + o_grad), k, s, nullptr, nullptr,
                                nullptr);
}
