// codec.cu -- stand-alone Kahan split/merge and u16 state pack/unpack kernels.
//
// Split/merge: the bf16 weight is the upper half of the fp32 master and the residual the 16
// low bits bf16 clips, so the pair restores the bit-identical f32 ("Kahan summation for
// Adafactor-optimized Flux FFT", sd-scripts PR #2159, first comment).
// Pack/unpack: scaled, biased, pow()-companded uint16 moments ("Amazing Flux FFT quality on a
// 5090", sd-scripts PR #2187, second post); constants fixed by this engine (see lmopt.h).
// These are HBM-bound grid-stride kernels with 128-bit accesses where every buffer allows it.
#include "internal.h"

namespace lmo {
namespace {

__global__ void __launch_bounds__(kThreads) k_split(const float* __restrict__ src,
                                                    uint16_t* __restrict__ hi,
                                                    uint16_t* __restrict__ lo, int64_t n, bool vec) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n >> 3;
        for (int64_t i = i0; i < nv; i += stride) {
            float4 a = ld_stream(reinterpret_cast<const float4*>(src) + 2 * i);
            float4 b = ld_stream(reinterpret_cast<const float4*>(src) + 2 * i + 1);
            uint32_t x[8] = {__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z),
                             __float_as_uint(a.w), __float_as_uint(b.x), __float_as_uint(b.y),
                             __float_as_uint(b.z), __float_as_uint(b.w)};
            uint4 h, l;
            h.x = (x[0] >> 16) | (x[1] & 0xFFFF0000u);
            h.y = (x[2] >> 16) | (x[3] & 0xFFFF0000u);
            h.z = (x[4] >> 16) | (x[5] & 0xFFFF0000u);
            h.w = (x[6] >> 16) | (x[7] & 0xFFFF0000u);
            l.x = (x[0] & 0xFFFFu) | (x[1] << 16);
            l.y = (x[2] & 0xFFFFu) | (x[3] << 16);
            l.z = (x[4] & 0xFFFFu) | (x[5] << 16);
            l.w = (x[6] & 0xFFFFu) | (x[7] << 16);
            st_stream(reinterpret_cast<uint4*>(hi) + i, h);
            st_stream(reinterpret_cast<uint4*>(lo) + i, l);
        }
        done = nv << 3;
    }
    for (int64_t i = done + i0; i < n; i += stride) {
        uint32_t b = __float_as_uint(src[i]);
        hi[i] = (uint16_t)(b >> 16);
        lo[i] = (uint16_t)(b & 0xFFFFu);
    }
}

__global__ void __launch_bounds__(kThreads) k_merge(const uint16_t* __restrict__ hi,
                                                    const uint16_t* __restrict__ lo,
                                                    float* __restrict__ dst, int64_t n, bool vec) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n >> 3;
        for (int64_t i = i0; i < nv; i += stride) {
            uint4 h = ld_stream(reinterpret_cast<const uint4*>(hi) + i);
            uint4 l = ld_stream(reinterpret_cast<const uint4*>(lo) + i);
            float4 a, b;
            a.x = __uint_as_float((h.x << 16) | (l.x & 0xFFFFu));
            a.y = __uint_as_float((h.x & 0xFFFF0000u) | (l.x >> 16));
            a.z = __uint_as_float((h.y << 16) | (l.y & 0xFFFFu));
            a.w = __uint_as_float((h.y & 0xFFFF0000u) | (l.y >> 16));
            b.x = __uint_as_float((h.z << 16) | (l.z & 0xFFFFu));
            b.y = __uint_as_float((h.z & 0xFFFF0000u) | (l.z >> 16));
            b.z = __uint_as_float((h.w << 16) | (l.w & 0xFFFFu));
            b.w = __uint_as_float((h.w & 0xFFFF0000u) | (l.w >> 16));
            st_stream(reinterpret_cast<float4*>(dst) + 2 * i, a);
            st_stream(reinterpret_cast<float4*>(dst) + 2 * i + 1, b);
        }
        done = nv << 3;
    }
    for (int64_t i = done + i0; i < n; i += stride)
        dst[i] = __uint_as_float(((uint32_t)hi[i] << 16) | (uint32_t)lo[i]);
}

// Pass 1 of pack: max of |x| (signed) or x (unsigned) as fp32 bit patterns into *scale_bits.
__global__ void __launch_bounds__(kThreads) k_absmax_f32(const float* __restrict__ src, int64_t n,
                                                         uint32_t* scale_bits) {
    __shared__ uint32_t red[32];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t mx[1] = {0u};
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        mx[0] = max(mx[0], __float_as_uint(src[i]) & 0x7FFFFFFFu);
    block_max_u32<1>(mx, red);
    if (threadIdx.x == 0 && mx[0] != 0u) atomicMax(scale_bits, mx[0]);
}

// Pass 2 of pack: encode with the scale found by pass 1.
__global__ void __launch_bounds__(kThreads) k_encode(const float* __restrict__ src,
                                                     uint16_t* __restrict__ codes, int64_t n,
                                                     const float* scale, int is_signed) {
    const float s = *scale;
    const CodecK c = codec_consts(s, s);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        float x = src[i];
        codes[i] = (uint16_t)(is_signed ? enc_m(x, c.rm) : enc_v(__fsqrt_rn(x), c.rv));
    }
}

__global__ void __launch_bounds__(kThreads) k_decode(const uint16_t* __restrict__ codes,
                                                     float* __restrict__ dst, int64_t n,
                                                     const float* scale, int is_signed) {
    const float s = *scale;
    const CodecK c = codec_consts(s, s);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = is_signed ? dec_m(codes[i], c.qm) : dec_v(codes[i], c.qv);
}

}  // namespace

int launch_kahan_split(const float* src, uint16_t* hi, uint16_t* lo, int64_t n, cudaStream_t s) {
    bool vec = is_aligned(src, 16) && is_aligned(hi, 16) && is_aligned(lo, 16);
    k_split<<<grid_for((n + 7) / 8), kThreads, 0, s>>>(src, hi, lo, n, vec);
    return check_cuda(cudaGetLastError(), "optim_kahan_split launch");
}

int launch_kahan_merge(const uint16_t* hi, const uint16_t* lo, float* dst, int64_t n, cudaStream_t s) {
    bool vec = is_aligned(dst, 16) && is_aligned(hi, 16) && is_aligned(lo, 16);
    k_merge<<<grid_for((n + 7) / 8), kThreads, 0, s>>>(hi, lo, dst, n, vec);
    return check_cuda(cudaGetLastError(), "optim_kahan_merge launch");
}

int launch_state_pack(const float* src, uint16_t* codes, float* scale, int64_t n, int is_signed,
                      cudaStream_t s) {
    int rc = check_cuda(cudaMemsetAsync(scale, 0, sizeof(float), s), "state_pack_u16 memset");
    if (rc) return rc;
    k_absmax_f32<<<grid_for(n), kThreads, 0, s>>>(src, n, reinterpret_cast<uint32_t*>(scale));
    rc = check_cuda(cudaGetLastError(), "state_pack_u16 absmax launch");
    if (rc) return rc;
    k_encode<<<grid_for(n), kThreads, 0, s>>>(src, codes, n, scale, is_signed);
    return check_cuda(cudaGetLastError(), "state_pack_u16 encode launch");
}

int launch_state_unpack(const uint16_t* codes, const float* scale, float* dst, int64_t n,
                        int is_signed, cudaStream_t s) {
    k_decode<<<grid_for(n), kThreads, 0, s>>>(codes, dst, n, scale, is_signed);
    return check_cuda(cudaGetLastError(), "state_unpack_u16 launch");
}

}  // namespace lmo
