// adan.cu -- fused Adan step ("a cpu-offloading version of ADAN ... four optimizer parameters
// for each model parameter", "Amazing Flux FFT quality on a 5090", sd-scripts PR #2187, fourth
// post; Algorithm 1 of the linked Adan paper).  States per element: m, v, n (fp32 planes of one
// buffer) and the previous bf16 gradient.  One pass per element; the weight is stored with the
// Kahan residual, stochastically rounded, or round-to-nearest.  38 bytes per element per step.
//   d = g - g_prev;  m = fma(1-b1, m, b1 g);  v = fma(1-b2, v, b2 d);  c = fma(1-b2, d, g)
//   n = fma(1-b3, n, b3 (c c));  u = fma(1-b2, v, m);  w = (w - lr (u / (sqrt(n) + eps))) / (1 + lr wd)
// Step 1 starts from m = g, v = 0, n = g^2; step 2 sets v = d (the paper's initialisation).
#include "internal.h"

namespace lmo {
namespace {

struct AdanPrm {
    float lr, b1, omb1, b2, omb2, b3, omb3, eps, inv_decay;
    int32_t sr;
    int64_t step;
    uint64_t seed;
};

__device__ __forceinline__ void philox4x64_10(uint64_t& c0, uint64_t& c1, uint64_t& c2, uint64_t& c3,
                                              uint64_t k0, uint64_t k1) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
}
__device__ __forceinline__ uint32_t sr_lane(const AdanPrm& k, uint32_t tensor, int64_t i) {
    uint64_t c0 = (uint64_t)i >> 4, c1 = (uint64_t)k.step, c2 = 0, c3 = 0;
    philox4x64_10(c0, c1, c2, c3, k.seed, tensor);
    const int lane = (int)(i & 15);
    const uint64_t wsel = lane < 4 ? c0 : (lane < 8 ? c1 : (lane < 12 ? c2 : c3));
    return (uint32_t)(wsel >> (16 * (lane & 3))) & 0xFFFFu;
}

__device__ __forceinline__ float adan_elem(const AdanPrm& k, float w, float g, float gp, float& m, float& v, float& n) {
    const float d = __fsub_rn(g, gp);
    if (k.step == 1) {
        m = g;
        v = 0.0f;
        n = __fmul_rn(g, g);
    } else {
        m = __fmaf_rn(k.omb1, m, __fmul_rn(k.b1, g));
        v = k.step == 2 ? d : __fmaf_rn(k.omb2, v, __fmul_rn(k.b2, d));
        const float c = __fmaf_rn(k.omb2, d, g);
        n = __fmaf_rn(k.omb3, n, __fmul_rn(k.b3, __fmul_rn(c, c)));
    }
    const float den = __fadd_rn(__fsqrt_rn(n), k.eps);
    const float u = __fmaf_rn(k.omb2, v, m);
    return __fmul_rn(__fsub_rn(w, __fmul_rn(k.lr, __fdiv_rn(u, den))), k.inv_decay);
}

__global__ void __launch_bounds__(kThreads) k_adan_step(NadamLaunch L, AdanPrm k) {
    __shared__ uint32_t red[32];
    const Chunk c = L.chunks[blockIdx.x];
    const TensorRec t = L.tensors[c.tensor];
    const uint16_t* __restrict__ g = L.grads[c.tensor];
    const bool has_res = (t.flags & kFlagRes) != 0;
    const int64_t n = t.numel;
    const int64_t start = (int64_t)c.index * kChunk;
    const int64_t end = min(n, start + kChunk);
    float* __restrict__ mp = static_cast<float*>(t.m);
    float* __restrict__ vp = mp + n;
    float* __restrict__ np_ = mp + 2 * n;
    uint16_t* __restrict__ gprev = static_cast<uint16_t*>(t.v);
    uint16_t* __restrict__ w = t.w;
    uint16_t* __restrict__ res = t.res;
    uint32_t nf = 0u;
    for (int64_t i = start + threadIdx.x; i < end; i += kThreads) {
        const float w0 = has_res ? __uint_as_float(((uint32_t)w[i] << 16) | res[i]) : bf16_to_f32(w[i]);
        const uint32_t gb = __ldcs(g + i);
        float m = __ldcs(mp + i), v = __ldcs(vp + i), nn = __ldcs(np_ + i);
        const float w1 = adan_elem(k, w0, bf16_to_f32(gb), bf16_to_f32(__ldcs(gprev + i)), m, v, nn);
        __stcs(mp + i, m);
        __stcs(vp + i, v);
        __stcs(np_ + i, nn);
        __stcs(gprev + i, (uint16_t)gb);
        const uint32_t b = __float_as_uint(w1);
        uint32_t hi;
        if (has_res) {
            hi = b >> 16;
            res[i] = (uint16_t)(b & 0xFFFFu);
        } else if (k.sr) {
            const uint32_t r = sr_lane(k, c.tensor, i);
            hi = ((b & 0x7F800000u) == 0x7F800000u) ? (b >> 16) : ((b + r) >> 16);
        } else {
            hi = rne_bf16(w1);
        }
        w[i] = (uint16_t)hi;
        nf = max(nf, hi & 0x7FFFu);
    }
    uint32_t r[1] = {nf >= 0x7F80u ? 1u : 0u};
    block_max_u32<1>(r, red);
    if (threadIdx.x == 0 && r[0]) atomicAdd(L.nonfinite, 1ull);
}

}  // namespace

int launch_adan_step(const NadamLaunch& L, const AdanScalars& s, cudaStream_t stream) {
    AdanPrm k{s.lr, s.b1, s.omb1, s.b2, s.omb2, s.b3, s.omb3, s.eps, s.inv_decay, s.sr, s.step, s.seed};
    if (L.n_chunks_total == 0) return OPTIM_OK;
    k_adan_step<<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
    return check_cuda(cudaGetLastError(), "adan step launch");
}

}  // namespace lmo
