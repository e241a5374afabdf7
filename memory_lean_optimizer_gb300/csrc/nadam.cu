// nadam.cu -- multi-tensor fused NAdam(W)/Adam step with Kahan residual and u16 moments.
//
// Two kernels per group call, each one CTA per chunk of the group's chunk table:
//  K1 k_grad_absmax : G = max|g| per u16-state tensor (the bound the encoder's scale needs before
//                     the step's moments exist); also clears the slots the step will accumulate.
//  K2 k_nadam_step  : per element, in one pass: merge (w_bf16, res) -> fp32 master, decode m, v,
//                     moment EMAs, decoupled decay, bias-corrected (Nesterov) update, split,
//                     re-encode, and the per-tensor maxima that bound the next step's scales.
// Sources: "Kahan summation for Adafactor-optimized Flux FFT" (sd-scripts PR #2159, first
// comment: the 16 clipped low bits restore the bit-identical f32); "Amazing Flux FFT quality on
// a 5090" (sd-scripts PR #2187: NAdam(W) first post, u16 scaled/biased/pow()-companded moments
// and the 4096-element fp32 rule second post, moments used only as storage third post).
//
// Per element the order of operations is (fma = one rounding):
//   w  = f32(hi<<16 | lo);  g = f32(g_bf16<<16)
//   m  = fma(b1, m0, (1-b1)*g);  v = fma(b2, v0, (1-b2)*(g*g))
//   w  = fma(-(lr*wd), w, w)                              (decoupled decay only)
//   sv = sqrt(v);  den = fma(sv, k2, eps);  num = fma(c_m, m, c_g*g);  w = fma(-lr, num/den, w)
//   (hi, lo) = split(w);  codes = enc_m(m), enc_v(sv) with the per-tensor codec constants
// with S_m = fma(b1, A_m(prev), (1-b1)*G), S_v = fma(b2, A_v(prev), (1-b2)*G*G) per tensor.
//
// Memory: 18 bytes per u16-state element per step (read w, res, g, m, v; write w, res, m, v),
// 26 bytes per fp32-state element, plus 2 bytes of K1's gradient read.  All accesses are
// 128-bit and coalesced when a tensor's buffers are 16-byte aligned.
#include "internal.h"

namespace lmo {
namespace {

struct Prm {
    float lr, b1, omb1, b2, omb2, eps, lr_wd, c_m, c_g, k2;
    int32_t decoupled;
    int32_t sr;           // stochastic rounding of tensors without a residual
    uint64_t step;
    PhiloxKey key;        // stochastic rounding: the generator's key schedule for the seed
};

// Random 16-bit lanes for the 8 elements i0 .. i0+7 (i0 % 8 == 0) of tensor `tensor`; word j
// holds lanes 2j (low half) and 2j+1.
__device__ __forceinline__ void sr_lanes8(const Prm& k, uint32_t tensor, int64_t i0, uint32_t (&r)[4]) {
    sr_block8(k.key, k.step, tensor, i0, r);
}
__device__ __forceinline__ uint32_t sr_lane1(const Prm& k, uint32_t tensor, int64_t i) {
    return sr_lane1(k.key, k.step, tensor, i);
}

// ------------------------------------------------------------------------------------ K1
// Per tensor max |g| (as the bf16 magnitude bits, atomicMax'ed into this step's slot) and, per
// chunk, whether its gradients hold an exact zero.  A resident grid of CTAs walks the group's
// u16-state chunks (CTA b takes chunks b, b + grid, ...): every thread issues all of its 128-bit
// loads of a chunk at once, and no CTA is launched per chunk, which matters for groups of many
// small tensors (hundreds of thousands of chunks).
constexpr int kK1Warps = kThreads / 32;
constexpr int kK1CtasPerSm = 4;   // 256-thread CTAs resident per SM (<= 64 registers per thread)

// One chunk of the pre-pass (every thread of the CTA).  red: 2 * kK1Warps words of shared memory.
__device__ __forceinline__ void k1_chunk(const NadamLaunch& L, int parity, int64_t ci, uint32_t* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = parity, q = parity ^ 1;
    const Chunk c = L.chunks[ci];
    const int64_t numel = L.tensors[c.tensor].numel;
    const uint16_t* __restrict__ g = L.grads[c.tensor];
    ScaleRec* sr = L.scales + c.tensor;
    if (c.index == 0 && threadIdx.x == 0) {
        sr->a_m[p] = 0u;   // this step's maxima accumulate here
        sr->a_v[p] = 0u;
        sr->g[q] = 0u;     // next step's gradient max accumulates here
    }
    const int64_t start = (int64_t)c.index * L.chunk;
    const int64_t end = min(numel, start + L.chunk);
    uint32_t mx = 0u;
    // exact zeros: a 16-bit magnitude t (bit 15 clear) is zero iff t - 1 sets bit 15; the
    // borrow into the upper half matters only when the lower half is zero, which is flagged anyway
    uint32_t zb = 0u;
    auto scan = [&](uint32_t x) {
        const uint32_t t = x & 0x7FFF7FFFu;
        zb |= t - 0x00010001u;
        return t;
    };
    auto scan4 = [&](const uint4& x) {
        mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(scan(x.x), scan(x.y)), __vmaxu2(scan(x.z), scan(x.w))));
    };
    int64_t done = start;
    if (aligned16(g)) {
        const int nv = (int)((end - start) >> 3);   // <= kChunkU16 / 8 = 16 * kThreads vectors
        const uint4* gv = reinterpret_cast<const uint4*>(g + start);
        constexpr int kLoads = (int)(kChunkU16 / 8 / kThreads);
        if (nv == kLoads * kThreads) {               // a whole chunk: all of a thread's loads in flight
            uint4 x[kLoads];
#pragma unroll
            for (int u = 0; u < kLoads; ++u) x[u] = __ldcg(gv + threadIdx.x + kThreads * u);
#pragma unroll
            for (int u = 0; u < kLoads; ++u) scan4(x[u]);
        } else {
            for (int i = threadIdx.x; i < nv; i += kThreads) scan4(__ldcg(gv + i));
        }
        done = start + ((int64_t)nv << 3);
    }
    mx = max(mx & 0xFFFFu, mx >> 16);
    for (int64_t i = done + threadIdx.x; i < end; i += kThreads) {
        const uint32_t t = g[i] & 0x7FFFu;
        mx = max(mx, t);
        if (t == 0u) zb |= 0x8000u;
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    const uint32_t zero = __reduce_or_sync(0xFFFFFFFFu, (zb & 0x80008000u) ? 1u : 0u);
    if (lane == 0) {
        red[warp] = mx;
        red[kK1Warps + warp] = zero;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, lane < kK1Warps ? red[lane] : 0u);
        const uint32_t z = __reduce_or_sync(0xFFFFFFFFu, lane < kK1Warps ? red[kK1Warps + lane] : 0u);
        if (lane == 0) {
            if (m != 0u) atomicMax(&sr->g[p], m << 16);
            L.zero_chunk[ci] = (uint8_t)z;
        }
    }
}

__global__ void __launch_bounds__(kThreads, kK1CtasPerSm) k_grad_absmax(NadamLaunch L, int parity) {
    __shared__ uint32_t red[2][2 * kK1Warps];   // by chunk parity: one barrier per chunk suffices
    int buf = 0;
    for (int64_t ci = blockIdx.x; ci < L.n_chunks_large; ci += gridDim.x, buf ^= 1) k1_chunk(L, parity, ci, red[buf]);
}

// ------------------------------------------------------------------------------------ K2
// Square root and quotient: kGuard selects the forms that keep exact zeros out of the library
// routines' special-value branch (same results; used where exact-zero gradients occur).
template <bool kGuard>
__device__ __forceinline__ float sqrt_k(float x) { return kGuard ? sqrt_rn_z(x) : __fsqrt_rn(x); }
template <bool kGuard>
__device__ __forceinline__ float div_k(float a, float b) { return kGuard ? div_rn_z(a, b) : __fdiv_rn(a, b); }

// One element: w, g fp32; m, v in: decoded (or fp32) moments, out: new moments; sv = sqrt(v).
template <bool kGuard>
__device__ __forceinline__ float elem(const Prm& k, float w, float g, float& m, float& v, float& sv) {
    m = __fmaf_rn(k.b1, m, __fmul_rn(k.omb1, g));
    v = __fmaf_rn(k.b2, v, __fmul_rn(k.omb2, __fmul_rn(g, g)));
    if (k.decoupled) w = __fmaf_rn(-k.lr_wd, w, w);
    sv = sqrt_k<kGuard>(v);
    const float den = __fmaf_rn(sv, k.k2, k.eps);
    const float num = __fmaf_rn(k.c_m, m, __fmul_rn(k.c_g, g));
    return __fmaf_rn(-k.lr, div_k<kGuard>(num, den), w);
}

// Packed fp32 pairs: __fmul2_rn / __fadd2_rn round each component exactly as the scalar _rn
// operation, so the paired decode and encode below give the same bits as the scalar helpers.
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Weight words in/out for two elements packed in 32-bit words W (bf16 weights) and R (residuals).
__device__ __forceinline__ void unpack_w(uint32_t W, uint32_t R, bool has_res, float& w0, float& w1) {
    w0 = __uint_as_float(has_res ? __byte_perm(R, W, 0x5410) : (W << 16));
    w1 = __uint_as_float(has_res ? __byte_perm(R, W, 0x7632) : (W & 0xFFFF0000u));
}
// rnd: two random 16-bit lanes (low half for w0) when stochastic rounding applies, else unused.
__device__ __forceinline__ void pack_w(float w0, float w1, bool has_res, bool sr, uint32_t rnd, uint32_t& W,
                                       uint32_t& R) {
    const uint32_t b0 = __float_as_uint(w0), b1 = __float_as_uint(w1);
    if (has_res) {
        W = pack_hi16(b0, b1);
        R = pack_lo16(b0, b1);
    } else if (sr) {
        W = pack_lo16(sr_bf16(w0, rnd & 0xFFFFu), sr_bf16(w1, rnd >> 16));
    } else {
        W = pack_lo16(rne_bf16(w0), rne_bf16(w1));
    }
}

struct Codec {
    CodecK dec, enc;
};

// Two u16-state elements.  am/av: running max |m|, max v (NaN skipped); nf: running max of the
// bf16 weight magnitudes (>= 0x7F80 in either half means a non-finite weight).
template <bool kGuard>
__device__ __forceinline__ void step2_u16(const Prm& k, const Codec& cd, bool has_res, bool sr, uint32_t rnd,
                                          uint32_t& W, uint32_t& R, uint32_t G, uint32_t& M, uint32_t& V,
                                          float& am, float& av, uint32_t& nf) {
    float2 w;
    unpack_w(W, R, has_res, w.x, w.y);
    // decode, as dec_m_field / dec_v_field, in pairs: t = (c - 32768) qm, m = t|t|;
    // z = c qv, v = (z z)(z z)  (codes to fp32 by the 2^23 mantissa trick)
    const float2 cm = make_float2(__uint_as_float(__byte_perm(M, 0x4B000000u, 0x7610)),
                                  __uint_as_float(__byte_perm(M, 0x4B000000u, 0x7632)));
    const float2 cv = make_float2(__uint_as_float(__byte_perm(V, 0x4B000000u, 0x7610)),
                                  __uint_as_float(__byte_perm(V, 0x4B000000u, 0x7632)));
    const float2 t = __fmul2_rn(__fadd2_rn(cm, f2(-8421376.0f)), f2(cd.dec.qm));
    float2 m = make_float2(__fmul_rn(t.x, fabsf(t.x)), __fmul_rn(t.y, fabsf(t.y)));
    const float2 z = __fmul2_rn(__fadd2_rn(cv, f2(-8388608.0f)), f2(cd.dec.qv));
    const float2 z2 = __fmul2_rn(z, z);
    float2 v = __fmul2_rn(z2, z2);
    float2 sv;
    w.x = elem<kGuard>(k, w.x, __uint_as_float(G << 16), m.x, v.x, sv.x);
    w.y = elem<kGuard>(k, w.y, __uint_as_float(G & 0xFFFF0000u), m.y, v.y, sv.y);
    pack_w(w.x, w.y, has_res, sr, rnd, W, R);
    // encode, as enc_m_bits / enc_v_bits, with the scaling multiply and the rounding add paired
    const float2 ym = make_float2(copysignf(fminf(sqrt_k<kGuard>(__fmul_rn(fabsf(m.x), cd.enc.rm)), 32767.0f), m.x),
                                  copysignf(fminf(sqrt_k<kGuard>(__fmul_rn(fabsf(m.y), cd.enc.rm)), 32767.0f), m.y));
    const float2 em = __fadd2_rn(f2(12615680.0f), ym);
    const float2 xv = __fmul2_rn(sv, f2(cd.enc.rv));
    const float2 yv = make_float2(fminf(sqrt_k<kGuard>(xv.x), 65535.0f), fminf(sqrt_k<kGuard>(xv.y), 65535.0f));
    const float2 ev = __fadd2_rn(f2(12582912.0f), yv);
    M = pack_lo16(__float_as_uint(em.x), __float_as_uint(em.y));
    V = pack_lo16(__float_as_uint(ev.x), __float_as_uint(ev.y));
    am = fmaxf(am, fmaxf(fabsf(m.x), fabsf(m.y)));
    av = fmaxf(av, fmaxf(v.x, v.y));
    nf = __vmaxu2(nf, W & 0x7FFF7FFFu);
}

// Two fp32-state elements (numel <= 4096).
__device__ __forceinline__ void step2_f32(const Prm& k, bool has_res, bool sr, uint32_t rnd, uint32_t& W,
                                          uint32_t& R, uint32_t G, float& m0, float& m1, float& v0, float& v1,
                                          uint32_t& nf) {
    float w0, w1, s0, s1;
    unpack_w(W, R, has_res, w0, w1);
    w0 = elem<true>(k, w0, __uint_as_float(G << 16), m0, v0, s0);
    w1 = elem<true>(k, w1, __uint_as_float(G & 0xFFFF0000u), m1, v1, s1);
    pack_w(w0, w1, has_res, sr, rnd, W, R);
    nf = __vmaxu2(nf, W & 0x7FFF7FFFu);
}

// i0: index of the first of the 8 elements (for the stochastic-rounding lanes).  kSR: the
// stochastic-rounding variant (compiled separately so the residual path carries none of it).
template <bool kSR, bool kGuard>
__device__ __forceinline__ void step8_u16(const Prm& k, const Codec& cd, bool has_res, const uint32_t (&r)[4],
                                          uint4& W, uint4& R, const uint4& G, uint4& M, uint4& V,
                                          float& am, float& av, uint32_t& nf) {
    const bool sr = kSR && !has_res;
    step2_u16<kGuard>(k, cd, has_res, sr, r[0], W.x, R.x, G.x, M.x, V.x, am, av, nf);
    step2_u16<kGuard>(k, cd, has_res, sr, r[1], W.y, R.y, G.y, M.y, V.y, am, av, nf);
    step2_u16<kGuard>(k, cd, has_res, sr, r[2], W.z, R.z, G.z, M.z, V.z, am, av, nf);
    step2_u16<kGuard>(k, cd, has_res, sr, r[3], W.w, R.w, G.w, M.w, V.w, am, av, nf);
}

template <bool kSR>
__device__ __forceinline__ void step8_f32(const Prm& k, bool has_res, uint32_t tensor, int64_t i0, uint4& W,
                                          uint4& R, const uint4& G, float4 (&M)[2], float4 (&V)[2], uint32_t& nf) {
    const bool sr = kSR && !has_res;
    uint32_t r[4] = {0u, 0u, 0u, 0u};
    if (sr) sr_lanes8(k, tensor, i0, r);
    step2_f32(k, has_res, sr, r[0], W.x, R.x, G.x, M[0].x, M[0].y, V[0].x, V[0].y, nf);
    step2_f32(k, has_res, sr, r[1], W.y, R.y, G.y, M[0].z, M[0].w, V[0].z, V[0].w, nf);
    step2_f32(k, has_res, sr, r[2], W.z, R.z, G.z, M[1].x, M[1].y, V[1].x, V[1].y, nf);
    step2_f32(k, has_res, sr, r[3], W.w, R.w, G.w, M[1].z, M[1].w, V[1].z, V[1].w, nf);
}

// The u16-state 128-bit path of one chunk (nv vectors of 8 elements starting at element `start`).
template <bool kSR, bool kGuard>
__device__ __forceinline__ void u16_vectors(const Prm& k, const Codec& cd, bool has_res, uint32_t tensor, int64_t start,
                                            int nv, uint4* wv, uint4* rv, const uint4* gv, uint4* mv, uint4* vv,
                                            float& am, float& av, uint32_t& nf) {
    // nv <= chunk / 8 <= kChunkU16 / 8: 32-bit vector indices within the chunk
    const bool sr = kSR && !has_res;
    // two independent 8-element groups per iteration, kThreads vectors apart: ten 128-bit
    // loads in flight (one generator call per group under stochastic rounding).
    int p = threadIdx.x;
    for (; p + kThreads < nv; p += 2 * kThreads) {
        const int i = p, i1 = p + kThreads;
        uint4 W0 = ld_stream(wv + i), W1 = ld_stream(wv + i1);
        uint4 R0 = has_res ? ld_stream(rv + i) : make_uint4(0, 0, 0, 0);
        uint4 R1 = has_res ? ld_stream(rv + i1) : make_uint4(0, 0, 0, 0);
        uint4 G0 = ld_stream(gv + i), G1 = ld_stream(gv + i1);
        uint4 M0 = ld_stream(mv + i), M1 = ld_stream(mv + i1);
        uint4 V0 = ld_stream(vv + i), V1 = ld_stream(vv + i1);
        uint32_t ra[4] = {0u, 0u, 0u, 0u}, rb[4] = {0u, 0u, 0u, 0u};
        if (sr) sr_lanes8(k, tensor, start + 8 * (int64_t)i, ra);
        step8_u16<kSR, kGuard>(k, cd, has_res, ra, W0, R0, G0, M0, V0, am, av, nf);
        st_stream(wv + i, W0);
        if (has_res) st_stream(rv + i, R0);
        st_stream(mv + i, M0);
        st_stream(vv + i, V0);
        if (sr) sr_lanes8(k, tensor, start + 8 * (int64_t)i1, rb);
        step8_u16<kSR, kGuard>(k, cd, has_res, rb, W1, R1, G1, M1, V1, am, av, nf);
        st_stream(wv + i1, W1);
        if (has_res) st_stream(rv + i1, R1);
        st_stream(mv + i1, M1);
        st_stream(vv + i1, V1);
    }
    // remaining vectors one at a time
    for (int i = p; i < nv; i += kThreads) {
        uint4 W0 = ld_stream(wv + i);
        uint4 R0 = has_res ? ld_stream(rv + i) : make_uint4(0, 0, 0, 0);
        uint4 G0 = ld_stream(gv + i), M0 = ld_stream(mv + i), V0 = ld_stream(vv + i);
        uint32_t ra[4] = {0u, 0u, 0u, 0u};
        if (sr) sr_lanes8(k, tensor, start + 8 * (int64_t)i, ra);
        step8_u16<kSR, kGuard>(k, cd, has_res, ra, W0, R0, G0, M0, V0, am, av, nf);
        st_stream(wv + i, W0);
        if (has_res) st_stream(rv + i, R0);
        st_stream(mv + i, M0);
        st_stream(vv + i, V0);
    }
}

// kFull: the group's chunk is kChunkU16 (every group but small ones), known at compile time.
// One chunk of the update (every thread of the CTA).  red: 3 * 32 words of shared memory.
template <bool kSR, bool kFull>
__device__ __forceinline__ void k2_chunk(const NadamLaunch& L, const Prm& k, int parity, int64_t ci, uint32_t* red) {
    const Chunk c = L.chunks[ci];
    const TensorRec t = L.tensors[c.tensor];
    const uint16_t* __restrict__ g = L.grads[c.tensor];
    const int p = parity, q = parity ^ 1;
    const bool small = (t.flags & kFlagSmall) != 0;
    const bool has_res = (t.flags & kFlagRes) != 0;
    const int64_t chunk = kFull ? kChunkU16 : L.chunk;
    const int64_t start = (int64_t)c.index * chunk;
    const int64_t end = min(t.numel, start + chunk);

    Codec cd{};
    ScaleRec* sr = L.scales + c.tensor;
    if (!small) {
        const float a_m = __uint_as_float(sr->a_m[q]), a_v = __uint_as_float(sr->a_v[q]);
        const float G = __uint_as_float(__ldcg(&sr->g[p]));
        const float s_m = __fmaf_rn(k.b1, a_m, __fmul_rn(k.omb1, G));
        const float s_v = __fmaf_rn(k.b2, a_v, __fmul_rn(k.omb2, __fmul_rn(G, G)));
        cd.dec = codec_consts(sr->s_m[q], sr->s_v[q]);
        cd.enc = codec_consts(s_m, s_v);
        if (c.index == 0 && threadIdx.x == 0) {
            sr->s_m[p] = s_m;
            sr->s_v[p] = s_v;
        }
    }

    float am = 0.f, av = 0.f;
    uint32_t nf = 0u;
    uint16_t* __restrict__ w = t.w;
    uint16_t* __restrict__ res = t.res;
    const bool vec = aligned16(w) && (!has_res || aligned16(res)) && aligned16(t.m) &&
                     aligned16(t.v) && aligned16(g);
    int64_t done = start;
    if (vec) {
        const int64_t nv = (end - start) >> 3;
        uint4* wv = reinterpret_cast<uint4*>(w + start);
        uint4* rv = has_res ? reinterpret_cast<uint4*>(res + start) : nullptr;
        const uint4* gv = reinterpret_cast<const uint4*>(g + start);
        if (!small) {
            uint4* mv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(t.m) + start);
            uint4* vv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(t.v) + start);
            // exact-zero gradients in this chunk (seen by the pre-pass): the zero-guarded
            // arithmetic, else the plain one (a branch taken by the whole CTA)
            if (L.zero_chunk == nullptr || __ldcg(L.zero_chunk + ci))
                u16_vectors<kSR, true>(k, cd, has_res, c.tensor, start, (int)nv, wv, rv, gv, mv, vv, am, av, nf);
            else
                u16_vectors<kSR, false>(k, cd, has_res, c.tensor, start, (int)nv, wv, rv, gv, mv, vv, am, av, nf);
        } else {
            float4* mv = reinterpret_cast<float4*>(static_cast<float*>(t.m) + start);
            float4* vv = reinterpret_cast<float4*>(static_cast<float*>(t.v) + start);
            for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
                uint4 W0 = ld_stream(wv + i);
                uint4 R0 = has_res ? ld_stream(rv + i) : make_uint4(0, 0, 0, 0);
                uint4 G0 = ld_stream(gv + i);
                float4 M[2] = {ld_stream(mv + 2 * i), ld_stream(mv + 2 * i + 1)};
                float4 V[2] = {ld_stream(vv + 2 * i), ld_stream(vv + 2 * i + 1)};
                step8_f32<kSR>(k, has_res, c.tensor, start + 8 * i, W0, R0, G0, M, V, nf);
                st_stream(wv + i, W0);
                if (has_res) st_stream(rv + i, R0);
                st_stream(mv + 2 * i, M[0]);
                st_stream(mv + 2 * i + 1, M[1]);
                st_stream(vv + 2 * i, V[0]);
                st_stream(vv + 2 * i + 1, V[1]);
            }
        }
        done = start + (nv << 3);
    }
    // element-by-element: ragged tail, or the whole chunk when a buffer is not 16-byte aligned
    for (int64_t i = done + threadIdx.x; i < end; i += kThreads) {
        const float w0 = has_res ? __uint_as_float(((uint32_t)w[i] << 16) | res[i]) : bf16_to_f32(w[i]);
        float m, v, sv;
        if (small) {
            m = static_cast<float*>(t.m)[i];
            v = static_cast<float*>(t.v)[i];
        } else {
            m = dec_m(static_cast<uint16_t*>(t.m)[i], cd.dec.qm);
            v = dec_v(static_cast<uint16_t*>(t.v)[i], cd.dec.qv);
        }
        const float w1 = elem<true>(k, w0, bf16_to_f32(g[i]), m, v, sv);
        const uint32_t b = __float_as_uint(w1);
        const uint32_t hi = has_res ? (b >> 16) : (kSR ? sr_bf16(w1, sr_lane1(k, c.tensor, i)) : rne_bf16(w1));
        w[i] = (uint16_t)hi;
        if (has_res) res[i] = (uint16_t)(b & 0xFFFFu);
        nf = max(nf, hi & 0x7FFFu);
        if (small) {
            static_cast<float*>(t.m)[i] = m;
            static_cast<float*>(t.v)[i] = v;
        } else {
            static_cast<uint16_t*>(t.m)[i] = (uint16_t)enc_m(m, cd.enc.rm);
            static_cast<uint16_t*>(t.v)[i] = (uint16_t)enc_v(sv, cd.enc.rv);
            am = fmaxf(am, fabsf(m));
            av = fmaxf(av, v);
        }
    }

    // per-tensor maxima for the next step's scales; one count per chunk with a non-finite weight
    uint32_t r[3] = {__float_as_uint(am), __float_as_uint(av), (max(nf & 0xFFFFu, nf >> 16) >= 0x7F80u) ? 1u : 0u};
    block_max_u32<3>(r, red);
    if (threadIdx.x == 0) {
        if (!small) {
            if (r[0]) atomicMax(&sr->a_m[p], r[0]);
            if (r[1]) atomicMax(&sr->a_v[p], r[1]);
        }
        if (r[2]) atomicAdd(L.nonfinite, 1ull);
    }
}

template <bool kSR, bool kFull>
__global__ void __launch_bounds__(kThreads, 4) k_nadam_step(NadamLaunch L, Prm k, int parity) {
    __shared__ uint32_t red[3 * 32];
    k2_chunk<kSR, kFull>(L, k, parity, blockIdx.x, red);
}

// ------------------------------------------------------------------------------------ one launch
// A group whose chunks all fit on the GPU at once (a cooperative launch, one CTA per chunk) steps
// in one kernel: the pre-pass of the CTA's chunk, a grid-wide barrier (the per-tensor gradient
// maxima are then complete), the update of the chunk.  It saves the second launch and its gap,
// which dominate a step of a small group (1024 x 1024: two launches of a few microseconds of
// work each).  The barrier counter only grows: each call adds the grid size and waits for the
// running total the host expects (compared modulo 2^32).  The wait is bounded (about a second);
// running out counts as a non-finite chunk, and the update proceeds.
constexpr long kBarrierSpin = 1L << 20;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <bool kSR>
__global__ void __launch_bounds__(kThreads, 4) k_nadam_fused(NadamLaunch L, Prm k, int parity, unsigned* bar,
                                                             unsigned target) {
    __shared__ uint32_t red[3 * 32];
    const int64_t ci = blockIdx.x;
    if (ci < L.n_chunks_large) k1_chunk(L, parity, ci, red);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(bar, 1u);
        unsigned v = ld_acquire_u32(bar);
        unsigned ns = 32;
        for (long it = 0; (int)(v - target) < 0 && it < kBarrierSpin; ++it) {
            __nanosleep(ns);
            ns = ns < 1024 ? 2 * ns : ns;
            v = ld_acquire_u32(bar);
        }
        if ((int)(v - target) < 0) atomicAdd(L.nonfinite, 1ull);
    }
    __syncthreads();
    k2_chunk<kSR, false>(L, k, parity, ci, red);
}

// ------------------------------------------------------------------------------------ f24
// f24 moments: the upper 24 bits of the fp32 moment (the f24 format of sd-scripts PR #2187,
// third post: fp32 cut to its top three bytes, eight mantissa bits more than bf16), stored as a
// plane of n upper 16-bit words followed by a plane of n bytes (bits 8..15; helpers in
// common.cuh).  Storage only: the update runs on the decoded fp32 values, and
// no scale (hence no gradient pre-pass) is needed.  22 bytes per element per step.

template <bool kSR>
__device__ __forceinline__ void step8_f24(const Prm& k, bool has_res, uint32_t tensor, int64_t i0, uint4& W, uint4& R,
                                          const uint4& G, uint4& MH, uint2& ML, uint4& VH, uint2& VL, uint32_t& nf) {
    const bool sr = kSR && !has_res;
    uint32_t rnd[4] = {0u, 0u, 0u, 0u};
    if (sr) sr_lanes8(k, tensor, i0, rnd);
    uint32_t* w32 = reinterpret_cast<uint32_t*>(&W);
    uint32_t* r32 = reinterpret_cast<uint32_t*>(&R);
    const uint32_t* g32 = reinterpret_cast<const uint32_t*>(&G);
    uint32_t* mh = reinterpret_cast<uint32_t*>(&MH);
    uint32_t* vh = reinterpret_cast<uint32_t*>(&VH);
    const uint32_t ml[2] = {ML.x, ML.y}, vl[2] = {VL.x, VL.y};
    uint32_t mb[8], vb[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float w0, w1, s0, s1;
        unpack_w(w32[j], r32[j], has_res, w0, w1);
        const uint32_t lm = ml[j >> 1] >> (16 * (j & 1)), lv = vl[j >> 1] >> (16 * (j & 1));
        float m0 = f24_value(mh[j] & 0xFFFFu, lm & 0xFFu), m1 = f24_value(mh[j] >> 16, (lm >> 8) & 0xFFu);
        float v0 = f24_value(vh[j] & 0xFFFFu, lv & 0xFFu), v1 = f24_value(vh[j] >> 16, (lv >> 8) & 0xFFu);
        w0 = elem<true>(k, w0, __uint_as_float(g32[j] << 16), m0, v0, s0);
        w1 = elem<true>(k, w1, __uint_as_float(g32[j] & 0xFFFF0000u), m1, v1, s1);
        pack_w(w0, w1, has_res, sr, rnd[j], w32[j], r32[j]);
        nf = __vmaxu2(nf, w32[j] & 0x7FFF7FFFu);
        mb[2 * j] = __float_as_uint(m0);
        mb[2 * j + 1] = __float_as_uint(m1);
        vb[2 * j] = __float_as_uint(v0);
        vb[2 * j + 1] = __float_as_uint(v1);
        mh[j] = pack_hi16(mb[2 * j], mb[2 * j + 1]);
        vh[j] = pack_hi16(vb[2 * j], vb[2 * j + 1]);
    }
    ML.x = pack_byte1(mb[0], mb[1], mb[2], mb[3]);
    ML.y = pack_byte1(mb[4], mb[5], mb[6], mb[7]);
    VL.x = pack_byte1(vb[0], vb[1], vb[2], vb[3]);
    VL.y = pack_byte1(vb[4], vb[5], vb[6], vb[7]);
}

template <bool kSR>
__global__ void __launch_bounds__(kThreads, 4) k_nadam_f24(NadamLaunch L, Prm k) {
    __shared__ uint32_t red[32];
    const Chunk c = L.chunks[blockIdx.x];
    const TensorRec t = L.tensors[c.tensor];
    const uint16_t* __restrict__ g = L.grads[c.tensor];
    const bool small = (t.flags & kFlagSmall) != 0;
    const bool has_res = (t.flags & kFlagRes) != 0;
    const int64_t n = t.numel;
    const int64_t start = (int64_t)c.index * L.chunk;
    const int64_t end = min(n, start + L.chunk);
    uint32_t nf = 0u;
    uint16_t* __restrict__ w = t.w;
    uint16_t* __restrict__ res = t.res;
    int64_t done = start;
    if (!small) {
        uint16_t* mhi = static_cast<uint16_t*>(t.m);
        uint16_t* vhi = static_cast<uint16_t*>(t.v);
        // The byte plane starts at 2n rounded up to 16 bytes, so that every tensor's planes are
        // 16-byte aligned together and ragged sizes keep the 128-bit path.
        uint8_t* mlo = static_cast<uint8_t*>(t.m) + f24_lo_offset(n);
        uint8_t* vlo = static_cast<uint8_t*>(t.v) + f24_lo_offset(n);
        const bool vec = aligned16(w) && (!has_res || aligned16(res)) && aligned16(g) && aligned16(mhi) &&
                         aligned16(vhi) && ((reinterpret_cast<uintptr_t>(mlo) | reinterpret_cast<uintptr_t>(vlo)) & 7u) == 0u;
        if (vec) {
            const int64_t nv = (end - start) >> 3;
            uint4* wv = reinterpret_cast<uint4*>(w + start);
            uint4* rv = has_res ? reinterpret_cast<uint4*>(res + start) : nullptr;
            const uint4* gv = reinterpret_cast<const uint4*>(g + start);
            uint4* mhv = reinterpret_cast<uint4*>(mhi + start);
            uint4* vhv = reinterpret_cast<uint4*>(vhi + start);
            uint2* mlv = reinterpret_cast<uint2*>(mlo + start);
            uint2* vlv = reinterpret_cast<uint2*>(vlo + start);
            for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
                uint4 W0 = ld_stream(wv + i);
                uint4 R0 = has_res ? ld_stream(rv + i) : make_uint4(0, 0, 0, 0);
                uint4 G0 = ld_stream(gv + i), MH = ld_stream(mhv + i), VH = ld_stream(vhv + i);
                uint2 ML = __ldcs(mlv + i), VL = __ldcs(vlv + i);
                step8_f24<kSR>(k, has_res, c.tensor, start + 8 * i, W0, R0, G0, MH, ML, VH, VL, nf);
                st_stream(wv + i, W0);
                if (has_res) st_stream(rv + i, R0);
                st_stream(mhv + i, MH);
                st_stream(vhv + i, VH);
                __stcs(mlv + i, ML);
                __stcs(vlv + i, VL);
            }
            done = start + (nv << 3);
        }
        for (int64_t i = done + threadIdx.x; i < end; i += kThreads) {
            const float w0 = has_res ? __uint_as_float(((uint32_t)w[i] << 16) | res[i]) : bf16_to_f32(w[i]);
            float m = f24_value(mhi[i], mlo[i]), v = f24_value(vhi[i], vlo[i]), sv;
            const float w1 = elem<true>(k, w0, bf16_to_f32(g[i]), m, v, sv);
            const uint32_t b = __float_as_uint(w1);
            const uint32_t hi = has_res ? (b >> 16) : (kSR ? sr_bf16(w1, sr_lane1(k, c.tensor, i)) : rne_bf16(w1));
            w[i] = (uint16_t)hi;
            if (has_res) res[i] = (uint16_t)(b & 0xFFFFu);
            nf = max(nf, hi & 0x7FFFu);
            const uint32_t mb = __float_as_uint(m), vb = __float_as_uint(v);
            mhi[i] = (uint16_t)(mb >> 16);
            vhi[i] = (uint16_t)(vb >> 16);
            mlo[i] = (uint8_t)(mb >> 8);
            vlo[i] = (uint8_t)(vb >> 8);
        }
    } else {
        float* mf = static_cast<float*>(t.m);
        float* vf = static_cast<float*>(t.v);
        for (int64_t i = start + threadIdx.x; i < end; i += kThreads) {
            const float w0 = has_res ? __uint_as_float(((uint32_t)w[i] << 16) | res[i]) : bf16_to_f32(w[i]);
            float m = mf[i], v = vf[i], sv;
            const float w1 = elem<true>(k, w0, bf16_to_f32(g[i]), m, v, sv);
            const uint32_t b = __float_as_uint(w1);
            const uint32_t hi = has_res ? (b >> 16) : (kSR ? sr_bf16(w1, sr_lane1(k, c.tensor, i)) : rne_bf16(w1));
            w[i] = (uint16_t)hi;
            if (has_res) res[i] = (uint16_t)(b & 0xFFFFu);
            nf = max(nf, hi & 0x7FFFu);
            mf[i] = m;
            vf[i] = v;
        }
    }
    uint32_t r[1] = {(max(nf & 0xFFFFu, nf >> 16) >= 0x7F80u) ? 1u : 0u};
    block_max_u32<1>(r, red);
    if (threadIdx.x == 0 && r[0]) atomicAdd(L.nonfinite, 1ull);
}

// ------------------------------------------------------------------------------------ scale exchange
// The codec scale of a tensor split across ranks needs the maxima over all of its slices: the
// step's gradient maximum G (slot p, from K1) and the previous step's moment maxima A_m, A_v
// (slot q).  Gather copies them per tensor into three consecutive floats (non-negative values,
// so a MAX reduction of the floats is a MAX of the bit patterns); scatter writes them back.
__global__ void k_scales_gather(const ScaleRec* sc, float* buf, int n, int parity) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int p = parity, q = parity ^ 1;
    buf[3 * i] = __uint_as_float(sc[i].g[p]);
    buf[3 * i + 1] = __uint_as_float(sc[i].a_m[q]);
    buf[3 * i + 2] = __uint_as_float(sc[i].a_v[q]);
}
__global__ void k_scales_scatter(ScaleRec* sc, const float* buf, int n, int parity) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int p = parity, q = parity ^ 1;
    sc[i].g[p] = __float_as_uint(buf[3 * i]);
    sc[i].a_m[q] = __float_as_uint(buf[3 * i + 1]);
    sc[i].a_v[q] = __float_as_uint(buf[3 * i + 2]);
}

}  // namespace

int launch_nadam_prepass(const NadamLaunch& L, const NadamScalars& s, cudaStream_t stream) {
    if (L.f24 || L.n_chunks_large == 0) return OPTIM_OK;   // f24 moments need no scale
    // at most the resident CTAs, each taking the same number of chunks (no partial last round)
    const int64_t cap = (int64_t)sm_count() * kK1CtasPerSm;
    const int64_t per = (L.n_chunks_large + cap - 1) / cap;
    const int64_t grid = (L.n_chunks_large + per - 1) / per;
    k_grad_absmax<<<(unsigned)grid, kThreads, 0, stream>>>(L, s.parity);
    return check_cuda(cudaGetLastError(), "grad absmax launch");
}

int nadam_fused_capacity(bool sr) {
    static int cache[2][256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    int& c = cache[sr ? 1 : 0][dev];
    if (c == 0) {
        int per_sm = 0, coop = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        const cudaError_t e = sr ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_nadam_fused<true>, kThreads, 0)
                                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_nadam_fused<false>, kThreads, 0);
        if (e != cudaSuccess) cudaGetLastError();
        c = (e == cudaSuccess && coop) ? per_sm * sm_count() : -1;
    }
    return c > 0 ? c : 0;
}

int launch_nadam_fused(const NadamLaunch& L, const NadamScalars& s, cudaStream_t stream, unsigned* bar,
                       unsigned target) {
    Prm k{s.lr, s.b1, s.omb1, s.b2, s.omb2, s.eps, s.lr_wd, s.c_m, s.c_g, s.k2, s.decoupled, s.sr, s.step, philox_key(s.seed)};
    NadamLaunch Lc = L;
    int parity = s.parity;
    void* args[] = {&Lc, &k, &parity, &bar, &target};
    const void* fn = s.sr ? reinterpret_cast<const void*>(k_nadam_fused<true>) : reinterpret_cast<const void*>(k_nadam_fused<false>);
    return check_cuda(cudaLaunchCooperativeKernel(fn, dim3((unsigned)L.n_chunks_total), dim3(kThreads), args, 0, stream),
                      "nadam one-launch step");
}

int launch_nadam_update(const NadamLaunch& L, const NadamScalars& s, cudaStream_t stream, cudaEvent_t mid) {
    Prm k{s.lr, s.b1, s.omb1, s.b2, s.omb2, s.eps, s.lr_wd, s.c_m, s.c_g, s.k2, s.decoupled, s.sr, s.step, philox_key(s.seed)};
    if (mid) {
        int rc = check_cuda(cudaEventRecord(mid, stream), "profile event");
        if (rc) return rc;
    }
    if (L.n_chunks_total == 0) return OPTIM_OK;
    if (L.f24) {
        if (k.sr) k_nadam_f24<true><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
        else k_nadam_f24<false><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k);
        return check_cuda(cudaGetLastError(), "nadam f24 step launch");
    }
    const bool full = L.chunk == kChunkU16;
    if (k.sr) {
        if (full) k_nadam_step<true, true><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k, s.parity);
        else k_nadam_step<true, false><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k, s.parity);
    } else {
        if (full) k_nadam_step<false, true><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k, s.parity);
        else k_nadam_step<false, false><<<L.n_chunks_total, kThreads, 0, stream>>>(L, k, s.parity);
    }
    return check_cuda(cudaGetLastError(), "nadam step launch");
}

int launch_scales_gather(const ScaleRec* sc, float* buf, int n, int parity, cudaStream_t stream) {
    if (n == 0) return OPTIM_OK;
    k_scales_gather<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(sc, buf, n, parity);
    return check_cuda(cudaGetLastError(), "scale gather launch");
}

int launch_scales_scatter(ScaleRec* sc, const float* buf, int n, int parity, cudaStream_t stream) {
    if (n == 0) return OPTIM_OK;
    k_scales_scatter<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(sc, buf, n, parity);
    return check_cuda(cudaGetLastError(), "scale scatter launch");
}

}  // namespace lmo
