// adan.cu -- fused Adan step (the page "Amazing Flux FFT quality on a 5090", sd-scripts PR #2187,
// fourth post, offers an offloaded Adan whose four states per parameter are kept small by
// compression; Algorithm 1 of the linked Adan paper).  States per element: m, v, n (fp32 planes of
// one buffer, or three f24 buffers in ADAN_F24 groups) and the previous bf16 gradient.  One pass
// per element; the weight is stored with the Kahan residual, stochastically rounded, or
// round-to-nearest.  38 bytes per element per step with fp32 states, 32 with f24 states.
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
    PhiloxKey key;        // stochastic rounding: the generator's key schedule for the seed
};

// Stochastic rounding draws from the same stream as the NAdam kernels (key, counter and lanes
// as described with philox4x32_10).
__device__ __forceinline__ void sr_block(const AdanPrm& k, uint32_t tensor, int64_t i, uint32_t (&r)[4]) {
    sr_block8(k.key, (uint64_t)k.step, tensor, i, r);
}
__device__ __forceinline__ uint32_t sr_lane(const AdanPrm& k, uint32_t tensor, int64_t i) {
    return sr_lane1(k.key, (uint64_t)k.step, tensor, i);
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
    const float den = __fadd_rn(sqrt_rn_z(n), k.eps);
    const float u = __fmaf_rn(k.omb2, v, m);
    return __fmul_rn(__fsub_rn(w, __fmul_rn(k.lr, div_rn_z(u, den))), k.inv_decay);
}

// Stores the updated weight (Kahan split, stochastic rounding or RNE); returns the bf16 word.
__device__ __forceinline__ uint32_t store_bits(float w1, bool has_res, bool sr, uint32_t rnd, uint32_t& lo) {
    const uint32_t b = __float_as_uint(w1);
    if (has_res) {
        lo = b & 0xFFFFu;
        return b >> 16;
    }
    lo = 0u;
    if (sr) return sr_bf16(w1, rnd);
    return rne_bf16(w1);
}

// The update of 8 consecutive elements held in registers: weights (W, R), gradients (G, GP) and
// the three states (ma, va, na, in place); returns the stored weight words in W, R.
template <bool kSR>
__device__ __forceinline__ void step8(const AdanPrm& k, bool has_res, uint32_t tensor, int64_t i0, uint4& W, uint4& R,
                                      const uint4& G, const uint4& GP, float (&ma)[8], float (&va)[8], float (&na)[8],
                                      uint32_t& nf) {
    uint32_t rnd[4] = {0u, 0u, 0u, 0u};
    if (kSR && !has_res) sr_block(k, tensor, i0, rnd);   // one block for these 8 elements
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&W);
    uint32_t* r32 = reinterpret_cast<uint32_t*>(&R);
    const uint32_t g32[4] = {G.x, G.y, G.z, G.w}, p32[4] = {GP.x, GP.y, GP.z, GP.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t wo = 0u, ro = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * q + h, sh = 16 * h;
            const uint32_t hw = (w32[q] >> sh) & 0xFFFFu, lw = (r32[q] >> sh) & 0xFFFFu;
            const float w0 = has_res ? __uint_as_float((hw << 16) | lw) : bf16_to_f32(hw);
            const float w1 = adan_elem(k, w0, bf16_to_f32((g32[q] >> sh) & 0xFFFFu),
                                       bf16_to_f32((p32[q] >> sh) & 0xFFFFu), ma[e], va[e], na[e]);
            uint32_t lo;
            const uint32_t hi = store_bits(w1, has_res, kSR, (rnd[q] >> sh) & 0xFFFFu, lo);
            wo |= hi << sh;
            ro |= lo << sh;
            nf = max(nf, hi & 0x7FFFu);
        }
        w32[q] = wo;
        r32[q] = ro;
    }
}

// 8 f24 values from an upper-word vector and a byte-plane pair, and back.
__device__ __forceinline__ void f24_unpack8(const uint4& H, const uint2& L, float (&x)[8]) {
    const uint32_t h[4] = {H.x, H.y, H.z, H.w}, l[2] = {L.x, L.y};
#pragma unroll
    for (int e = 0; e < 8; ++e)
        x[e] = f24_value((h[e >> 1] >> (16 * (e & 1))) & 0xFFFFu, (l[e >> 2] >> (8 * (e & 3))) & 0xFFu);
}
__device__ __forceinline__ void f24_pack8(const float (&x)[8], uint4& H, uint2& L) {
    uint32_t b[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) b[e] = __float_as_uint(x[e]);
    H = make_uint4(pack_hi16(b[0], b[1]), pack_hi16(b[2], b[3]), pack_hi16(b[4], b[5]), pack_hi16(b[6], b[7]));
    L = make_uint2(pack_byte1(b[0], b[1], b[2], b[3]), pack_byte1(b[4], b[5], b[6], b[7]));
}

// kSR: stochastic rounding of weights without a residual (a template flag so that the Philox
// state stays out of the register budget of the other variants).  kF24: the group keeps m, v
// and n of tensors above 4096 elements as three f24 buffers (upper words, padding, byte plane;
// buffer j at byte j * f24_stride(n)) instead of fp32 planes; smaller tensors keep fp32 planes.
template <bool kSR, bool kF24>
__global__ void __launch_bounds__(kThreads, 4) k_adan_step(NadamLaunch L, AdanPrm k) {
    __shared__ uint32_t red[32];
    const Chunk c = L.chunks[blockIdx.x];
    const TensorRec t = L.tensors[c.tensor];
    const uint16_t* __restrict__ g = L.grads[c.tensor];
    const bool has_res = (t.flags & kFlagRes) != 0;
    const bool f24 = kF24 && (t.flags & kFlagSmall) == 0;
    const int64_t n = t.numel;
    const int64_t start = (int64_t)c.index * L.chunk;
    const int64_t end = min(n, start + L.chunk);
    uint16_t* __restrict__ gprev = static_cast<uint16_t*>(t.v);
    uint16_t* __restrict__ w = t.w;
    uint16_t* __restrict__ res = t.res;
    uint32_t nf = 0u;
    // fp32 planes (plane stride n rounded up to 4 floats) or f24 buffers of the three states
    float* __restrict__ mp = static_cast<float*>(t.m);
    const int64_t plane = (n + 3) & ~int64_t(3);
    float* __restrict__ vp = mp + plane;
    float* __restrict__ np_ = mp + 2 * plane;
    uint8_t* const fb = static_cast<uint8_t*>(t.m);
    const int64_t fs = f24 ? f24_stride(n) : 0, flo = f24 ? f24_lo_offset(n) : 0;
    uint16_t* __restrict__ mh = reinterpret_cast<uint16_t*>(fb);
    uint16_t* __restrict__ vh = reinterpret_cast<uint16_t*>(fb + fs);
    uint16_t* __restrict__ nh = reinterpret_cast<uint16_t*>(fb + 2 * fs);
    uint8_t* __restrict__ ml = fb + flo;
    uint8_t* __restrict__ vl = fb + fs + flo;
    uint8_t* __restrict__ nl = fb + 2 * fs + flo;
    // 8 elements per thread per iteration with 128-bit accesses when every buffer is 16-byte
    // aligned (chunk starts are multiples of 8 elements; plane strides are multiples of 4 floats,
    // f24 strides and byte-plane offsets multiples of 16 bytes); the rest element by element
    const bool vec = aligned16(w) && (!has_res || aligned16(res)) && aligned16(g) && aligned16(gprev) &&
                     aligned16(mp);
    const int64_t vend = vec ? start + ((end - start) & ~int64_t(7)) : start;
    for (int64_t i = start + 8 * (int64_t)threadIdx.x; i < vend; i += 8 * kThreads) {
        uint4 W = ld_stream(reinterpret_cast<const uint4*>(w + i));
        uint4 R = has_res ? ld_stream(reinterpret_cast<const uint4*>(res + i)) : make_uint4(0, 0, 0, 0);
        const uint4 G = ld_stream(reinterpret_cast<const uint4*>(g + i));
        const uint4 GP = ld_stream(reinterpret_cast<const uint4*>(gprev + i));
        float ma[8], va[8], na[8];
        if (f24) {
            f24_unpack8(ld_stream(reinterpret_cast<const uint4*>(mh + i)), __ldcs(reinterpret_cast<const uint2*>(ml + i)), ma);
            f24_unpack8(ld_stream(reinterpret_cast<const uint4*>(vh + i)), __ldcs(reinterpret_cast<const uint2*>(vl + i)), va);
            f24_unpack8(ld_stream(reinterpret_cast<const uint4*>(nh + i)), __ldcs(reinterpret_cast<const uint2*>(nl + i)), na);
        } else {
            *reinterpret_cast<float4*>(ma) = ld_stream(reinterpret_cast<const float4*>(mp + i));
            *reinterpret_cast<float4*>(ma + 4) = ld_stream(reinterpret_cast<const float4*>(mp + i + 4));
            *reinterpret_cast<float4*>(va) = ld_stream(reinterpret_cast<const float4*>(vp + i));
            *reinterpret_cast<float4*>(va + 4) = ld_stream(reinterpret_cast<const float4*>(vp + i + 4));
            *reinterpret_cast<float4*>(na) = ld_stream(reinterpret_cast<const float4*>(np_ + i));
            *reinterpret_cast<float4*>(na + 4) = ld_stream(reinterpret_cast<const float4*>(np_ + i + 4));
        }
        step8<kSR>(k, has_res, c.tensor, i, W, R, G, GP, ma, va, na, nf);
        st_stream(reinterpret_cast<uint4*>(w + i), W);
        if (has_res) st_stream(reinterpret_cast<uint4*>(res + i), R);
        st_stream(reinterpret_cast<uint4*>(gprev + i), G);
        if (f24) {
            uint4 H;
            uint2 Lo;
            f24_pack8(ma, H, Lo);
            st_stream(reinterpret_cast<uint4*>(mh + i), H);
            __stcs(reinterpret_cast<uint2*>(ml + i), Lo);
            f24_pack8(va, H, Lo);
            st_stream(reinterpret_cast<uint4*>(vh + i), H);
            __stcs(reinterpret_cast<uint2*>(vl + i), Lo);
            f24_pack8(na, H, Lo);
            st_stream(reinterpret_cast<uint4*>(nh + i), H);
            __stcs(reinterpret_cast<uint2*>(nl + i), Lo);
        } else {
            st_stream(reinterpret_cast<float4*>(mp + i), *reinterpret_cast<const float4*>(ma));
            st_stream(reinterpret_cast<float4*>(mp + i + 4), *reinterpret_cast<const float4*>(ma + 4));
            st_stream(reinterpret_cast<float4*>(vp + i), *reinterpret_cast<const float4*>(va));
            st_stream(reinterpret_cast<float4*>(vp + i + 4), *reinterpret_cast<const float4*>(va + 4));
            st_stream(reinterpret_cast<float4*>(np_ + i), *reinterpret_cast<const float4*>(na));
            st_stream(reinterpret_cast<float4*>(np_ + i + 4), *reinterpret_cast<const float4*>(na + 4));
        }
    }
    for (int64_t i = vend + threadIdx.x; i < end; i += kThreads) {
        const float w0 = has_res ? __uint_as_float(((uint32_t)w[i] << 16) | res[i]) : bf16_to_f32(w[i]);
        const uint32_t gb = __ldcs(g + i);
        float m, v, nn;
        if (f24) {
            m = f24_value(mh[i], ml[i]);
            v = f24_value(vh[i], vl[i]);
            nn = f24_value(nh[i], nl[i]);
        } else {
            m = __ldcs(mp + i);
            v = __ldcs(vp + i);
            nn = __ldcs(np_ + i);
        }
        const float w1 = adan_elem(k, w0, bf16_to_f32(gb), bf16_to_f32(__ldcs(gprev + i)), m, v, nn);
        if (f24) {
            const uint32_t bm = __float_as_uint(m), bv = __float_as_uint(v), bn = __float_as_uint(nn);
            mh[i] = (uint16_t)(bm >> 16);
            ml[i] = (uint8_t)(bm >> 8);
            vh[i] = (uint16_t)(bv >> 16);
            vl[i] = (uint8_t)(bv >> 8);
            nh[i] = (uint16_t)(bn >> 16);
            nl[i] = (uint8_t)(bn >> 8);
        } else {
            __stcs(mp + i, m);
            __stcs(vp + i, v);
            __stcs(np_ + i, nn);
        }
        __stcs(gprev + i, (uint16_t)gb);
        uint32_t lo;
        const uint32_t hi = store_bits(w1, has_res, kSR, (kSR && !has_res) ? sr_lane(k, c.tensor, i) : 0u, lo);
        if (has_res) res[i] = (uint16_t)lo;
        w[i] = (uint16_t)hi;
        nf = max(nf, hi & 0x7FFFu);
    }
    uint32_t r[1] = {nf >= 0x7F80u ? 1u : 0u};
    block_max_u32<1>(r, red);
    if (threadIdx.x == 0 && r[0]) atomicAdd(L.nonfinite, 1ull);
}

}  // namespace

int launch_adan_step(const NadamLaunch& L, const AdanScalars& s, cudaStream_t stream) {
    AdanPrm k{s.lr, s.b1, s.omb1, s.b2, s.omb2, s.b3, s.omb3, s.eps, s.inv_decay, s.sr, s.step, philox_key(s.seed)};
    if (L.n_chunks_total == 0) return OPTIM_OK;
    if (L.f24) {
        if (s.sr) k_adan_step<true, true><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
        else k_adan_step<false, true><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
    } else {
        if (s.sr) k_adan_step<true, false><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
        else k_adan_step<false, false><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
    }
    return check_cuda(cudaGetLastError(), "adan step launch");
}

}  // namespace lmo
