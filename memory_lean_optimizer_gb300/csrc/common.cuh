// common.cuh -- device helpers and tables shared by the engine's kernels (sm_103a).
//
// Every floating-point operation on the state path is an explicit round-to-nearest intrinsic
// (__fmul_rn, __fadd_rn, __fsqrt_rn, __fdiv_rn, and __fmaf_rn where a fused multiply-add with
// one rounding is meant), which the compiler never fuses or reorders; the library is also built
// with --fmad=false.  The results are therefore the IEEE fp32 results of the operation order
// written here, on every run.
#pragma once

#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "../../include/lmopt.h"

namespace lmo {

constexpr int kThreads = 256;          // threads per CTA of the streaming kernels
constexpr int64_t kChunk = 16384;      // elements per CTA of the f24 and Adan kernels; multiple of 8
constexpr int64_t kChunkU16 = 32768;   // elements per CTA of NAdam u16 groups (pre-pass + update):
                                       // the update's per-chunk prologue (chunk, tensor and scale
                                       // records, codec constants) is shared by twice the elements
constexpr int64_t kChunkMin = 2048;    // smallest chunk a small group is cut into
constexpr int64_t kSmall = OPTIM_SMALL_NUMEL;

// Flags of a tensor record.
constexpr int32_t kFlagSmall = 1;      // fp32 moments (numel <= 4096)
constexpr int32_t kFlagRes = 2;        // has a Kahan residual

// One parameter tensor, as the kernels see it.  48 bytes.
struct TensorRec {
    uint16_t* w;
    uint16_t* res;
    void* m;
    void* v;
    int64_t numel;
    int32_t flags;
    int32_t pad;
};

// Per-tensor scale record of the u16 codec, double-buffered by step parity p:
// slot p is written by the step with parity p and read (as "previous") by the next step.
//   s_m, s_v : scales the codes were encoded with
//   a_m, a_v : max |m|, max v before encoding (fp32 bit patterns, atomicMax'ed)
//   g        : max |g| of the step's gradient (fp32 bit pattern of the bf16 magnitude)
struct ScaleRec {
    float s_m[2];
    float s_v[2];
    uint32_t a_m[2];
    uint32_t a_v[2];
    uint32_t g[2];
    uint32_t pad[6];
};
static_assert(sizeof(ScaleRec) == 64, "ScaleRec layout");

// One CTA's work item: elements [index*chunk, min(numel, (index+1)*chunk)) of a tensor, chunk the
// group's chunk size (kChunkU16 or kChunk by kind, or a smaller power of two for groups too small
// to fill the GPU).
struct Chunk {
    int32_t tensor;
    int32_t index;
};

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// IEEE square root and quotient with an exact-zero operand kept out of the library routines'
// special-value branch: a lane whose argument is zero computes on 1 instead and selects the
// exact answer (sqrt(+-0) = +-0; +-0 / b = +-0 for b > 0; any other b divides as usual).  Same
// results as __fsqrt_rn / __fdiv_rn; without it, exact-zero gradients (a few per warp) make
// whole warps diverge.
__device__ __forceinline__ float sqrt_rn_z(float x) {
    const bool z = x == 0.0f;
    const float r = __fsqrt_rn(z ? 1.0f : x);
    return z ? x : r;
}
__device__ __forceinline__ float div_rn_z(float a, float b) {
    const bool z = a == 0.0f && b > 0.0f;
    const float r = __fdiv_rn(z ? b : a, b);
    return z ? a : r;
}

// Round-to-nearest-even fp32 -> bf16 bits (store used when no residual is kept); NaN keeps
// its payload's upper bits with the quiet bit set.
__device__ __forceinline__ uint32_t rne_bf16(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0u) return (b >> 16) | 0x0040u;
    uint32_t up = b >> 16, rem = b & 0xFFFFu;
    up += (rem > 0x8000u || (rem == 0x8000u && (up & 1u))) ? 1u : 0u;
    return up & 0xFFFFu;
}

// ---- stochastic rounding -------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC 2011): four 32-bit counter words, ten rounds of two 32x32->64 multiplies; round r XORs in
// the key words k0 + r W0 and k1 + r W1 (Weyl sequence), precomputed here once per launch so
// that the rounds read them as kernel parameters.  Key (seed low, seed high); counter (b low,
// b high, tensor, step mod 2^32) for the 8-element block b = i / 8; element i takes 16-bit lane
// i mod 8 (word (i mod 8) / 2, low half for even i).
struct PhiloxKey {
    uint32_t k0[10], k1[10];
};
__host__ __device__ inline PhiloxKey philox_key(uint64_t seed) {
    PhiloxKey key;
    for (int r = 0; r < 10; ++r) {
        key.k0[r] = (uint32_t)seed + (uint32_t)r * 0x9E3779B9u;
        key.k1[r] = (uint32_t)(seed >> 32) + (uint32_t)r * 0xBB67AE85u;
    }
    return key;
}
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], const PhiloxKey& key) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)M0 * c[0], p1 = (uint64_t)M1 * c[2];
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ key.k0[r];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ key.k1[r];
        c[0] = n0;
        c[1] = (uint32_t)p1;
        c[2] = n2;
        c[3] = (uint32_t)p0;
    }
}
// The random words of the 8-element block holding element i (i need not be a multiple of 8).
__device__ __forceinline__ void sr_block8(const PhiloxKey& key, uint64_t step, uint32_t tensor, int64_t i,
                                          uint32_t (&r)[4]) {
    const uint64_t b = (uint64_t)i >> 3;
    r[0] = (uint32_t)b;
    r[1] = (uint32_t)(b >> 32);
    r[2] = tensor;
    r[3] = (uint32_t)step;
    philox4x32_10(r, key);
}
// Element i's 16 random bits.
__device__ __forceinline__ uint32_t sr_lane1(const PhiloxKey& key, uint64_t step, uint32_t tensor, int64_t i) {
    uint32_t r[4];
    sr_block8(key, step, tensor, i, r);
    const int lane = (int)(i & 7);
    const uint32_t wsel = lane < 2 ? r[0] : (lane < 4 ? r[1] : (lane < 6 ? r[2] : r[3]));
    return (wsel >> (16 * (lane & 1))) & 0xFFFFu;
}
// Stochastic rounding to bf16 bits: the 16 random bits are added below the kept half, which
// rounds the magnitude up with probability (dropped bits) / 2^16.  Infinities and NaNs are kept
// as they are (a NaN's all-ones payload would otherwise carry into the sign).
__device__ __forceinline__ uint32_t sr_bf16(float x, uint32_t r16) {
    const uint32_t b = __float_as_uint(x);
    return (b + (fabsf(x) < __int_as_float(0x7F800000) ? r16 : 0u)) >> 16;
}

// ---- u16 companded codec --------------------------------------------------------------
// Curve: exp_avg code = 32768 + sgn(m) rint(32767 (|m|/S)^(1/2)); exp_avg_sq code =
// rint(65535 (v/S)^(1/4)).  Scale and code step are folded into four per-tensor constants:
//   qm = sqrt(S_m)/32767, rm = 1/qm^2   (decode m = t|t|, t = (c-32768) qm; encode sqrt(|m| rm))
//   qv = S_v^(1/4)/65535, rv = 1/qv^2   (decode v = (z z)(z z), z = c qv; encode sqrt(sqrt(v) rv))
struct CodecK {
    float qm, rm, qv, rv;
};
__device__ __forceinline__ CodecK codec_consts(float s_m, float s_v) {
    CodecK c;
    c.qm = __fmul_rn(__fsqrt_rn(s_m), 1.0f / 32767.0f);
    c.rm = s_m > 0.0f ? fminf(__fdiv_rn(1.0f, __fmul_rn(c.qm, c.qm)), FLT_MAX) : 0.0f;
    c.qv = __fmul_rn(__fsqrt_rn(__fsqrt_rn(s_v)), 1.0f / 65535.0f);
    c.rv = s_v > 0.0f ? fminf(__fdiv_rn(1.0f, __fmul_rn(c.qv, c.qv)), FLT_MAX) : 0.0f;
    return c;
}

// Exact int -> float of a 16-bit field without the conversion unit: the field is placed in the
// mantissa of 2^23 and 2^23 is subtracted.  sel: 0x7610 for the low half of `word`, 0x7632 for
// the high half.
template <unsigned kSel>
__device__ __forceinline__ float u16_field_to_f32(uint32_t word, float minus) {
    return __fadd_rn(__uint_as_float(__byte_perm(word, 0x4B000000u, kSel)), minus);
}
// Decoded moments of the code in the low (kSel 0x7610) or high (0x7632) half of a word.
template <unsigned kSel>
__device__ __forceinline__ float dec_m_field(uint32_t word, float qm) {
    const float t = __fmul_rn(u16_field_to_f32<kSel>(word, -8421376.0f), qm);   // c - 32768
    return __fmul_rn(t, fabsf(t));
}
template <unsigned kSel>
__device__ __forceinline__ float dec_v_field(uint32_t word, float qv) {
    const float z = __fmul_rn(u16_field_to_f32<kSel>(word, -8388608.0f), qv);
    const float z2 = __fmul_rn(z, z);
    return __fmul_rn(z2, z2);
}
__device__ __forceinline__ float dec_m(uint32_t c, float qm) { return dec_m_field<0x7610>(c, qm); }
__device__ __forceinline__ float dec_v(uint32_t c, float qv) { return dec_v_field<0x7610>(c, qv); }

// Encoders return a float whose low 16 bits are the code: adding 1.5*2^23 (+32768 for the
// biased exp_avg code) rounds the clamped root to the nearest integer, ties to even, exactly as
// rint, and leaves it in the low mantissa bits.
__device__ __forceinline__ uint32_t enc_m_bits(float m, float rm) {
    const float y = fminf(sqrt_rn_z(__fmul_rn(fabsf(m), rm)), 32767.0f);
    return __float_as_uint(__fadd_rn(12615680.0f, copysignf(y, m)));
}
// sv = sqrt(v), shared with the update's denominator.
__device__ __forceinline__ uint32_t enc_v_bits(float sv, float rv) {
    const float y = fminf(sqrt_rn_z(__fmul_rn(sv, rv)), 65535.0f);
    return __float_as_uint(__fadd_rn(12582912.0f, y));
}
__device__ __forceinline__ uint32_t enc_m(float m, float rm) { return enc_m_bits(m, rm) & 0xFFFFu; }
__device__ __forceinline__ uint32_t enc_v(float sv, float rv) { return enc_v_bits(sv, rv) & 0xFFFFu; }

// Packs the low 16 bits of two words (element 0 low, element 1 high) / the high 16 bits.
__device__ __forceinline__ uint32_t pack_lo16(uint32_t e0, uint32_t e1) { return __byte_perm(e0, e1, 0x5410); }
__device__ __forceinline__ uint32_t pack_hi16(uint32_t e0, uint32_t e1) { return __byte_perm(e0, e1, 0x7632); }

// ---- f24 storage: the upper 24 bits of an fp32 value, as a plane of n upper 16-bit words,
// zero padding up to byte 2n rounded up to 16, then a plane of n bytes (bits 8..15) ----
__device__ __forceinline__ int64_t f24_lo_offset(int64_t n) { return (2 * n + 15) & ~(int64_t)15; }
// Bytes between consecutive f24 buffers of one allocation (Adan's m, v, n): the buffer's bytes
// rounded up to 16, so that every buffer starts 16-byte aligned.
__device__ __forceinline__ int64_t f24_stride(int64_t n) { return (f24_lo_offset(n) + n + 15) & ~(int64_t)15; }
__device__ __forceinline__ float f24_value(uint32_t hi16, uint32_t lo8) { return __uint_as_float((hi16 << 16) | (lo8 << 8)); }
// Bits 8..15 of four fp32 patterns, packed into one word (element 0 in the low byte).
__device__ __forceinline__ uint32_t pack_byte1(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
    return __byte_perm(__byte_perm(b0, b1, 0x0051), __byte_perm(b2, b3, 0x0051), 0x5410);
}

// ---- block reductions (kThreads threads) ----
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}
__device__ __forceinline__ float warp_sum_f32(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

// Max over the block of up to three values; result valid in thread 0.
template <int N>
__device__ __forceinline__ void block_max_u32(uint32_t (&v)[N], uint32_t* smem /* N*32 */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = warp_max_u32(v[i]);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) smem[i * 32 + warp] = v[i];
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            uint32_t x = lane < nw ? smem[i * 32 + lane] : 0u;
            v[i] = warp_max_u32(x);
        }
    }
}

// Streaming 128-bit loads and stores: data touched once per step, evict first.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

__device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;
}

}  // namespace lmo
