// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "common.cuh"

namespace lmo {

// True when the environment variable LMOPT_FAULT_INJECT equals `what` (host-side fault
// injection for the error-path tests: h2d, d2h, alloc, timeout).
bool fault_injected(const char* what);
// Records the thread-local error message and returns `code`.
int set_error(int code, const char* fmt, ...);
// OPTIM_OK if e == cudaSuccess, else records "<what>: <cuda message>" and returns OPTIM_ECUDA.
int check_cuda(cudaError_t e, const char* what);
// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();
// Grid for a grid-stride elementwise kernel over `units` work units of kThreads each.
unsigned grid_for(int64_t units);

inline bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- launchers (each returns OPTIM_OK or OPTIM_ECUDA after checking the launch) ----
int launch_kahan_split(const float* src, uint16_t* hi, uint16_t* lo, int64_t n, cudaStream_t s);
int launch_kahan_merge(const uint16_t* hi, const uint16_t* lo, float* dst, int64_t n, cudaStream_t s);
int launch_state_pack(const float* src, uint16_t* codes, float* scale, int64_t n, int is_signed,
                      cudaStream_t s);
int launch_state_unpack(const uint16_t* codes, const float* scale, float* dst, int64_t n,
                        int is_signed, cudaStream_t s);

// Per-step scalars of the NAdam/Adam kernel (host-computed: double, then one rounding).
struct NadamScalars {
    float lr, b1, omb1, b2, omb2, eps, lr_wd, c_m, c_g, k2;
    int32_t decoupled;
    int32_t parity;
    int32_t sr;        // stochastic rounding for tensors without a residual
    uint64_t seed;
    uint64_t step;
};

struct NadamLaunch {
    const TensorRec* tensors;
    const uint16_t* const* grads;
    ScaleRec* scales;
    const Chunk* chunks;
    unsigned long long* nonfinite;
    int32_t n_chunks_large;   // chunks of u16-state tensors come first
    int32_t n_chunks_total;
    int32_t f24;              // moments stored as f24 planes instead of u16 codes
    uint8_t* zero_chunk;      // per u16 chunk: the gradient pre-pass saw an exact zero (K2 then
                              // takes the zero-guarded arithmetic for that chunk)
    int64_t chunk;            // elements per chunk (a power of two, kChunkMin..kChunkU16)
};
// K1 (gradient maxima; nothing for f24 moments), then K2 (the update; `mid`, if not null, is
// recorded on the stream before it).  A step is both, in this order, on one stream.
int launch_nadam_prepass(const NadamLaunch& L, const NadamScalars& k, cudaStream_t s);
int launch_nadam_update(const NadamLaunch& L, const NadamScalars& k, cudaStream_t s, cudaEvent_t mid);
// The pre-pass and the update in one cooperative launch (one CTA per chunk), for groups whose
// chunks all fit on the GPU at once: nadam_fused_capacity() chunks at most (0: not available).
// bar: the group's barrier counter; target: its value once every CTA of this launch has arrived.
int nadam_fused_capacity(bool sr);
int launch_nadam_fused(const NadamLaunch& L, const NadamScalars& k, cudaStream_t s, unsigned* bar, unsigned target);
// Per tensor {G (this step), A_m, A_v (previous step)} to / from 3 consecutive floats.
int launch_scales_gather(const ScaleRec* sc, float* buf, int n, int parity, cudaStream_t s);
int launch_scales_scatter(ScaleRec* sc, const float* buf, int n, int parity, cudaStream_t s);

// Per-step scalars of the Adan kernel.
struct AdanScalars {
    float lr, b1, omb1, b2, omb2, b3, omb3, eps, inv_decay;
    int32_t sr;
    int64_t step;
    uint64_t seed;
};
int launch_adan_step(const NadamLaunch& L, const AdanScalars& k, cudaStream_t s);

}  // namespace lmo
