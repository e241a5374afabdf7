/*
 * lmopt.h -- C ABI of the GB300 fused optimizer-step engine (liblmopt.so).
 *
 * The engine performs the per-parameter optimizer step of memory-lean full fine-tuning:
 * a group of parameters is registered once, then "step this group" is called each time the
 * group's gradients are complete -- the granularity of the fused backward pass and of
 * optimizer groups ("Fused backward pass" commit, README, "Fused optimizer" and "Optimizer
 * groups" items).
 *
 * Conventions
 *  - Every function returns int: OPTIM_OK (0) or a negative OPTIM_E* code.  On error,
 *    optim_last_error() returns a thread-local message.  A failing call validates everything
 *    before its first launch, so weights and states are left untouched.
 *  - Device buffers are owned by the caller.  The library owns its group handle and the small
 *    device tables behind it (tensor table, chunk table, per-tensor scales), freed by
 *    optim_group_destroy.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  All work is
 *    enqueued asynchronously on it; only optim_group_create, optim_query_* and optim_set_*
 *    synchronise.  Calls on one group must be ordered by the caller (one stream, or events).
 *  - bf16 and uint16 buffers are arrays of 16-bit words and must be 2-byte aligned; fp32 buffers
 *    4-byte aligned.  16-byte alignment of every buffer of a tensor enables 128-bit accesses;
 *    other alignments take a slower element-by-element path with identical results.
 *  - All arithmetic is IEEE fp32, each operation rounded once to nearest-even: the update's
 *    a*b+c steps are fused multiply-adds (one rounding), nothing else is contracted.  The
 *    results are deterministic run to run.
 *  - Environment (read at each call): LMOPT_VERBOSE=1 prints one line per created group (see
 *    optim_group_create); LMOPT_FAULT_INJECT=h2d|d2h|alloc makes the offload path fail with
 *    OPTIM_ECUDA / OPTIM_ENOMEM before it enqueues anything, and =timeout makes every bounded
 *    host wait return OPTIM_ETIMEOUT at once (host-side tests of the error paths; nothing on the
 *    GPU is disturbed).
 */
#ifndef LMOPT_H
#define LMOPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    OPTIM_OK = 0,
    OPTIM_EINVAL = -1,     /* bad argument (NULL pointer, size, shape, hyper-parameter, step) */
    OPTIM_ECUDA = -2,      /* a CUDA runtime call or launch failed */
    OPTIM_ENOMEM = -3,     /* device or pinned host allocation failed */
    OPTIM_EALIGN = -4,     /* a buffer is not aligned to its element size */
    OPTIM_ETIMEOUT = -5,   /* a bounded host wait on a stream event ran out */
    OPTIM_ENONFINITE = -6, /* reserved for callers that turn a nonzero non-finite count into an error */
    OPTIM_ESTATE = -7      /* call not valid in the group's current state */
};

/* Tensors of this many elements or fewer keep fp32 moments instead of u16 codes (small tensors
 * skip the compact format and stay in f32, "Amazing Flux FFT quality on a 5090", sd-scripts
 * PR #2187, second post). */
#define OPTIM_SMALL_NUMEL 4096

typedef struct optim_group optim_group_t;

/* One parameter tensor of a group.
 *   w_bf16  : device, numel bf16 weights (the upper 16 bits of the fp32 master), in/out
 *   res_u16 : device, numel uint16 Kahan residuals (the 16 low bits bf16 drops), in/out, or
 *             NULL: no residual, the weight is stored round-to-nearest-even
 *   m, v    : kind NADAM: exp_avg / exp_avg_sq -- numel uint16 codes if numel > 4096, else
 *             numel fp32 values.
 *             kind FACTORED: ndim >= 2: m = row state fp32 [prod(shape[:-1])], v = column state
 *             fp32 [prod(shape[:-2]) * shape[-1]]; ndim == 1: m unused (NULL), v = full fp32
 *             second moment [numel].
 *   numel   : element count (0 allowed: the tensor is skipped)
 *   ndim, shape : logical shape, 1 <= ndim <= 4, product == numel (FACTORED groups factor the
 *             last two dims; NADAM groups ignore the shape).
 * All buffers must stay valid and unmoved for the life of the group. */
typedef struct {
    void* w_bf16;
    void* res_u16;
    void* m;
    void* v;
    int64_t numel;
    int32_t ndim;
    int32_t reserved;
    int64_t shape[4];
} optim_tensor_desc_t;

/* Group kinds.  NADAM_F24 is NADAM with f24 moment storage: the upper three bytes of each fp32
 * moment, truncated (the f24 format of "Amazing Flux FFT quality on a 5090", sd-scripts PR
 * #2187, third post: fp32 cut to its top three bytes, eight mantissa bits more than bf16).
 * Its m and v buffers (numel > 4096) hold L + numel bytes, L = 2*numel rounded up to a multiple of 16: numel uint16
 * upper words, padding up to byte L, then numel bytes of bits 8..15.  Buffers that start on a
 * 16-byte boundary take the 128-bit path whatever numel is.  No scale records and no gradient
 * pre-pass are involved; tensors of 4096 or fewer elements keep fp32 moments. */
enum {
    OPTIM_KIND_NADAM = 0,
    OPTIM_KIND_FACTORED = 1,
    OPTIM_KIND_NADAM_F24 = 2,
    OPTIM_KIND_ADAN = 3,
    OPTIM_KIND_ADAN_F24 = 4
};
/* ADAN groups: m -> fp32 [3*P] (planes m, v, n, each P = numel rounded up to a multiple of 4
 * floats, so that every plane of a 16-byte aligned buffer is 16-byte aligned and takes the
 * 128-bit path), v -> uint16 [numel] (previous bf16 gradient), all zero at creation.
 * ADAN_F24 groups keep Adan's three states in the f24 storage of NADAM_F24 (the page offering
 * the offloaded Adan, "Amazing Flux FFT quality on a 5090", sd-scripts PR #2187, fourth post,
 * names compression of its four states without fixing one): for numel > 4096, m holds three
 * f24 buffers of the NADAM_F24 layout -- m, v and n -- each padded to F = (L + numel) rounded up
 * to 16 bytes, buffer j at byte j*F (3F bytes); tensors of 4096 or fewer elements keep the fp32
 * planes of ADAN.  Storage only: the update computes on the decoded fp32 values.  v as ADAN.
 * 32 bytes per element per step instead of 38. */

/* Adam / NAdam(W) hyper-parameters ("(N)AdamW / Adan with fused backwards pass & CPU
 * offloading", sd-scripts PR #2187, first post: NAdamOffload, AdamOffload, NAdamWOffload).
 *   wd_mode  : 0 none, 1 decoupled (the "W" variants: w -= lr*wd*w before the update)
 *   nesterov : 0 Adam, 1 NAdam (Dozat's momentum schedule mu_t = beta1 (1 - 0.5*0.96^(t*psi)))
 *   momentum_decay : psi, 0.004 by default
 *   stochastic_rounding : 1 = tensors WITHOUT a residual store the new weight stochastically
 *             rounded to bf16 instead of round-to-nearest (sd-scripts' default alternative to
 *             Kahan summation, "Kahan summation for Adafactor-optimized Flux FFT", PR #2159, PR
 *             description): 16 random bits are added below the kept half.  The bits come from
 *             Philox4x32-10 (Salmon et al., SC 2011) with key (seed mod 2^32, seed / 2^32) and
 *             counter (b mod 2^32, b / 2^32, tensor index in the group, step mod 2^32) for the
 *             block b = element / 8, element i taking 16-bit lane i mod 8 (word (i mod 8) / 2, low
 *             half first); results are reproducible.
 *   seed     : key of the stochastic rounding */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int32_t wd_mode;
    int32_t nesterov;
    float momentum_decay;
    int32_t stochastic_rounding;
    uint64_t seed;
} optim_nadam_hparams_t;

/* Factored second-moment hyper-parameters (beta1 = 0: no exp_avg is read or written).
 *   mode 0 Adafactor ("Fused backward pass" commit, library/adafactor_fused.py,
 *          adafactor_step_param): beta2_t = 1 - t^decay_rate, eps1 added to g^2 before the means.
 *   mode 1 Prodigy ("more VRAM savings: no first moment and factored second moment",
 *          prodigy PR #25): constant beta2, EMAs weighted by d^2 (1-beta2), eps2 added after the
 *          EMA; the update's numerator is d g (Prodigy's first moment with beta1 = 0) and the
 *          step size d*lr.  d is hp->d, or, in a group attached to a Prodigy controller
 *          (optim_group_attach_prodigy), the controller's current estimate.
 *   clip_threshold : update clipping, u /= max(1, RMS(u)/clip_threshold)
 *   weight_decay   : decoupled, w += w * (-wd * lr_eff) before the update */
typedef struct {
    float lr, beta2, decay_rate, eps1, eps2, d, clip_threshold, weight_decay;
    int32_t mode;
} optim_factored_hparams_t;

/* Registers `n` tensors as one group (n >= 1) and allocates the group's device tables
 * (tensor table, chunk table, per-tensor scale records).  Synchronises (one upload).
 * All scale records start at zero; the u16 m codes must start at 32768 and v codes at 0 (the
 * zero point), fp32 moments and factored states at 0.  With the environment variable
 * LMOPT_VERBOSE=1 each created group prints one line to stderr (tensors, elements, state kind,
 * how many tensors keep a Kahan residual, the chunking), as the Kahan change of "Kahan summation
 * for Adafactor-optimized Flux FFT" reports on the console that it is active. */
int optim_group_create(const optim_tensor_desc_t* tensors, int32_t n, int32_t kind,
                       optim_group_t** out);
int optim_group_destroy(optim_group_t* group);

/* One fused NAdam(W)/Adam step of every tensor of a NADAM or NADAM_F24 group, in one pass per element:
 * rebuild the fp32 master from (w_bf16, res_u16), decode m and v, update the moments, apply
 * decoupled decay and the bias-corrected (Nesterov) update, split the master back into
 * (w_bf16, res_u16), re-encode m and v, and reduce the per-tensor maxima that bound the next
 * step's scales.  Before it, a pre-pass reduces max|g| per u16 tensor.
 * ("Kahan summation for Adafactor-optimized Flux FFT", sd-scripts PR #2159, first comment:
 * the 16 clipped low bits restore the bit-identical f32; PR #2187, second post: scaled,
 * biased, pow()-companded uint16 moments.)
 *   grads_bf16 : host array of n device pointers, one bf16 gradient per tensor, same order as at
 *                create (may change from call to call; unchanged pointers cost no upload)
 *   step       : 1 on the first call, then previous + 1; anything else is OPTIM_EINVAL
 * Two enqueued kernels (one if every tensor has 4096 or fewer elements, or if the group is small
 * enough for all of its 2048..32768-element chunks to run on the GPU at once: the pre-pass, a
 * grid-wide barrier and the update then form one cooperative launch, with the same results).
 * The barrier's wait is bounded (about a second); should it run out, the chunk is counted by
 * optim_query_nonfinite and the step's results are not to be trusted. */
int optim_step_nadam_kahan(optim_group_t* group, const void* const* grads_bf16, int64_t step,
                           const optim_nadam_hparams_t* hp, void* stream);
/* Kernel launches one step of the group enqueues with these hyper-parameters (NADAM groups: 1 or
 * 2, see optim_step_nadam_kahan; NADAM_F24, ADAN, ADAN_F24: 1; hp may be NULL for those).
 * OPTIM_EINVAL for FACTORED groups, whose launches depend on their waves. */
int optim_query_launches(optim_group_t* group, const optim_nadam_hparams_t* hp, int32_t* launches);

/* The same step in two calls, for a tensor split into slices across ranks (each rank's group
 * holds its slices as tensors).  The codec scale belongs to the whole tensor: it is bounded by
 * the maxima over all slices of max|g| (this step) and of the moment maxima (previous step), so
 * the ranks combine them between the gradient pre-pass and the update.  Splitting is otherwise
 * exact -- the update of an element depends only on its own values and the scale -- so slices
 * stepped this way are bit-identical to the unsplit tensor, provided every slice of a tensor of
 * more than 4096 elements has more than 4096 elements too (a slice of 4096 or fewer keeps fp32
 * moments, as a whole tensor of that size would).  The pages have no counterpart: their step
 * is per parameter on one GPU; this is the data-parallel form of the same step.
 *   begin    : validates, uploads gradient pointers, enqueues the pre-pass; if `exchange` (a device
 *              buffer of 3 floats per tensor, 4-byte aligned, caller-owned) is not NULL, copies
 *              into it, per tensor i, {max|g|, max|m| of the previous step, max v of the previous
 *              step} at [3i, 3i+1, 3i+2] (non-negative values; NaN if a gradient held NaN).
 *   (caller) : MAX all-reduce of `exchange` across the ranks holding slices of the same tensors
 *              (the same tensor order on every rank), on `stream` or ordered after it.
 *   end      : if `exchange` is not NULL, writes its values back, then enqueues the update.
 * Between begin and end the group accepts no other call that changes its state (OPTIM_ESTATE);
 * begin twice, or end without begin, is OPTIM_ESTATE.  optim_step_nadam_kahan is begin + end with
 * no exchange.  f24 groups have no scale: their exchange values are carried but unused. */
int optim_step_nadam_begin(optim_group_t* group, const void* const* grads_bf16, int64_t step,
                           const optim_nadam_hparams_t* hp, void* stream, float* exchange);
int optim_step_nadam_end(optim_group_t* group, const float* exchange, void* stream);

/* One factored-second-moment step (Adafactor / Prodigy with beta1 = 0) of a FACTORED group:
 * row and column EMAs of g^2 over the last two dims, rank-1 reconstruction
 * V_ij = R_i C_j / mean(R), update u = g / sqrt(V), RMS clipping, decoupled decay, Kahan split.
 * 1-D tensors keep a full second moment.  Arguments as optim_step_nadam_kahan.  A group larger
 * than one wave (96 MiB of gradients) is processed wave by wave, with consecutive waves on up to
 * three streams: `stream` and two streams owned by the group, which wait for the work already on
 * `stream` and which `stream` waits for before any later work -- to the caller the call is
 * ordered on `stream` as usual.  A group attached to a Prodigy controller also runs its
 * statistics on a fourth stream of its own, ordered the same way. */
int optim_step_factored(optim_group_t* group, const void* const* grads_bf16, int64_t step,
                        const optim_factored_hparams_t* hp, void* stream);

/* Single-tensor factored step that allocates nothing (the pages have no counterpart; this entry
 * exists for callers that cannot call cudaMalloc -- e.g. code whose device memory is entirely
 * owned by another allocator or fixed pool, or a long-running job that must not allocate once it
 * has been set up).  optim_step_factored allocates its scratch when the group is created; this
 * variant instead uses one fixed 32 MiB device array that the library holds on every GPU that
 * loads it, until the process exits.  The caller passes the tensor (weights, optional residual,
 * factored state, as in optim_tensor_desc_t for FACTORED groups) and its bf16 gradient; results
 * are identical to a FACTORED group holding just this tensor.  `step` is the caller's own
 * counter (>= 1; no sequence check).  A tensor whose scratch would exceed the array (about 3/64
 * byte per element of a matrix: some 7e8 elements) is rejected with OPTIM_EINVAL and a message
 * giving both sizes.
 * The first call on a device looks up the array's device address (once per device).  All calls
 * share the array and it keeps the previous call's contents (the call clears the parts that must
 * start at zero), so calls whose work overlaps on the GPU -- different streams without ordering,
 * or several host threads -- race: order them on one stream.  Calls no cudaMalloc, cudaFree or other allocating routine. */
int optim_step_factored_noalloc(const optim_tensor_desc_t* tensor, const void* grad_bf16, int64_t step,
                                const optim_factored_hparams_t* hp, void* stream);

/* ---- Prodigy's step-size estimate d over FACTORED groups (mode 1) ---------------------------
 * The pages discuss Prodigy's d (prodigy PR #25: d0, the numerator built from p - p0, "s, which
 * is the denominator in the calculation of d_hat", the EMAs scaled by d) without printing its
 * update; this follows the Adam form of Prodigy (Mishchenko, Defazio, "Prodigy: An Expeditiously
 * Adaptive Parameter-Free Learner", 2023) with beta1 = 0.  Over every tensor of every group
 * attached to one controller, a step k with d_k (the fp32 value of the controller's d) does,
 * before the group's update and with x the master weight before it:
 *     r   = beta3 r + lr d_k^2 sum_e g_e (p0_e - x_e),     s_e = beta3 s_e + fl(lr d_k^2) g_e
 * and optim_prodigy_end_step, after all attached groups have stepped, sets
 *     d_{k+1} = max(d_k, r / sum_e |s_e|)      (unchanged while the sum is 0).
 * The sums run over a subsample ("sliced", prodigy PR #22): the 64-element blocks of each
 * tensor's flat elements whose block index is a multiple of slice_p (1: every element).  p0 and
 * s hold the sampled elements in order, 64 per sampled block.  d, r and the step's partial sums
 * live in device memory: no call of a step synchronises. */
typedef struct optim_prodigy optim_prodigy_t;
/* d0 > 0 (the first d), 0 <= beta3 < 1 (Prodigy's default: sqrt(beta2)), slice_p >= 1. */
int optim_prodigy_create(double d0, float beta3, int32_t slice_p, optim_prodigy_t** out);
/* OPTIM_ESTATE while groups are attached (destroy them first). */
int optim_prodigy_destroy(optim_prodigy_t* pd);
/* Floats in each of a tensor's p0 and s buffers: 64 * ceil(ceil(numel / 64) / slice_p); -1 if
 * numel < 0 or slice_p < 1. */
int64_t optim_prodigy_slice_len(int64_t numel, int32_t slice_p);
/* Attaches a FACTORED group (between steps).  p0[i], s[i]: caller-owned fp32 DEVICE buffers of
 * optim_prodigy_slice_len(numel_i, slice_p) floats, 4-byte aligned, one pair per tensor, kept
 * alive while attached.  snapshot = 1: enqueued on `stream`, p0 takes the current master
 * weights at the sampled elements (0 past a tensor's end) and s is zeroed (the start of
 * training); snapshot = 0: the buffers are used as they are (resuming from a checkpoint that
 * saved them).  The group's later steps must use mode 1; hp->d is then ignored.  A group
 * attaches once. */
int optim_group_attach_prodigy(optim_group_t* group, optim_prodigy_t* pd, void* const* p0, void* const* s,
                               int32_t snapshot, void* stream);
/* Ends a step of the controller's groups: reduces the statistics the attached groups' steps
 * left (in a fixed order) and updates r and d.  Enqueued on `stream`, which must be ordered after
 * those steps (the same stream, or one that waits for them); groups not stepped add nothing. */
int optim_prodigy_end_step(optim_prodigy_t* pd, void* stream);
/* The same in two halves, for data-parallel processes that each step their own groups and share
 * one d: reduce writes this process's sums (sum over its groups of lr d^2 sum g (p0 - x), and
 * sum |s|) as 2 doubles to `partial` (DEVICE, 8-byte aligned) and clears the statistics; the
 * caller SUM-reduces the 2 doubles across processes (e.g. an all-reduce) and passes the totals
 * to finish, which updates r and d the same way on every process.  Both enqueued on `stream`. */
int optim_prodigy_reduce(optim_prodigy_t* pd, double* partial, void* stream);
int optim_prodigy_finish(optim_prodigy_t* pd, const double* total, void* stream);
/* Current d and r (synchronises the device); set them between steps, e.g. on checkpoint resume. */
int optim_prodigy_get(optim_prodigy_t* pd, double* d, double* r);
int optim_prodigy_set(optim_prodigy_t* pd, double d, double r);

/* Adan hyper-parameters (Algorithm 1 of the Adan paper linked by "Amazing Flux FFT quality on a
 * 5090", sd-scripts PR #2187, fourth post; beta weights the new term, as in the paper).
 * stochastic_rounding / seed as in optim_nadam_hparams_t (tensors without a residual). */
typedef struct {
    float lr, beta1, beta2, beta3, eps, weight_decay;
    int32_t stochastic_rounding;
    int32_t reserved;
    uint64_t seed;
} optim_adan_hparams_t;

/* One fused Adan step of an ADAN or ADAN_F24 group: d = g - g_prev, m, v, n EMAs, w = (w - lr (m + (1-b2) v) /
 * (sqrt(n) + eps)) / (1 + lr wd), Kahan split (or stochastic / nearest rounding), g_prev = g.
 * Step 1 starts from m = g, v = 0, n = g^2 and step 2 sets v = d.  Arguments as
 * optim_step_nadam_kahan; one enqueued kernel. */
int optim_step_adan(optim_group_t* group, const void* const* grads_bf16, int64_t step,
                    const optim_adan_hparams_t* hp, void* stream);

/* Encodes n fp32 moments into u16 codes with the engine's codec.  scale (device, 1 float) is
 * written with max|src| (is_signed = 1, exp_avg) or max src (is_signed = 0, exp_avg_sq); codes
 * are 32768 + sgn(x) rint(32767 sqrt(|x|/S)) or rint(65535 (x/S)^(1/4)).  Two kernels. */
int state_pack_u16(const float* src, uint16_t* codes, float* scale, int64_t n, int32_t is_signed,
                   void* stream);
/* Decodes n u16 codes with the device scale: S t|t|, t = (c-32768)/32767, or S z^4, z = c/65535. */
int state_unpack_u16(const uint16_t* codes, const float* scale, float* dst, int64_t n,
                     int32_t is_signed, void* stream);

/* fp32 <-> (bf16 upper half, uint16 lower half), bit-exact both ways.  hi/lo/src/dst device. */
int optim_kahan_split(const float* src, uint16_t* hi, uint16_t* lo, int64_t n, void* stream);
int optim_kahan_merge(const uint16_t* hi, const uint16_t* lo, float* dst, int64_t n, void* stream);

/* Per-tensor scale records after the last completed step, 4 floats per tensor in group order:
 * S_m, S_v (scales the stored codes were encoded with), A_m, A_v (max |m| and max v before
 * encoding).  host_out holds 4*n floats.  Synchronises the group's last stream. */
int optim_query_scales(optim_group_t* group, float* host_out);
/* Restores scale records (same layout) before the next step, e.g. on checkpoint resume. */
int optim_set_scales(optim_group_t* group, const float* host_in);
/* Step counter and NAdam momentum product (the product of mu_1..mu_t, kept in double). */
int optim_group_get_step(optim_group_t* group, int64_t* step, double* mu_product);
int optim_group_set_step(optim_group_t* group, int64_t step, double mu_product);
/* Non-finite detection: the number of (step, chunk) pairs in which an updated weight came out
 * NaN or infinite, summed over all steps so far (a chunk is up to 32768 elements of one tensor;
 * in FACTORED groups, one unit of the update kernel: a 128x256 tile, up to 2048 small matrices,
 * or up to 2048 elements of a 1-D tensor). */
int optim_query_nonfinite(optim_group_t* group, uint64_t* count);

/* ---- pinned-host offload of the states between steps --------------------------------------
 * The pages keep the optimizer states and Kahan residuals in CPU memory between steps and move
 * each parameter group's states in for its update and back out afterwards ("Amazing Flux FFT
 * quality on a 5090", sd-scripts PR #2187, first post, and its fourth post for Adan; "Kahan
 * summation for Adafactor-optimized Flux FFT", sd-scripts PR #2159, PR description).  NADAM,
 * NADAM_F24, ADAN and ADAN_F24 groups can be offloaded: their residuals and m, v buffers then
 * live in PINNED HOST memory, while weights, gradients and the per-tensor scale records stay on
 * the device.  Each step runs on a device staging slot: the copy-in (prefetch) must precede the
 * step, the copy-out (write-back) follows it; every dependency between them is a device-side
 * event wait, so the host never blocks.  Prefetching group k+1 and writing back group k-1 while
 * group k steps overlaps the copies with the kernels.  A group holds its slot from prefetch to
 * write-back; a prefetch takes the first free slot after the one taken last, and returns
 * OPTIM_ESTATE when every slot is held (at most n_slots groups hold slots at once).
 *
 * Two ways to attach a group:
 *   optim_group_attach_host (the per-group form): the caller gives one pinned buffer, the
 *     group's host image, and enqueues prefetch and write-back itself on copy streams of its
 *     choice; one copy per direction.  Staging slots come from the library's own ring on the
 *     group's device (three slots, sized to the largest attached group, freed with the last).
 *   optim_group_attach_offload (an engine the caller creates): the group's descriptors point at
 *     pinned host buffers; a step prefetches if the caller has not, and enqueues its own
 *     write-back on the engine's D2H stream. */
typedef struct optim_offload optim_offload_t;
int optim_offload_create(size_t slot_bytes, int32_t n_slots, optim_offload_t** out);
/* Waits (bounded) for the engine's copies, then frees it; OPTIM_ESTATE while groups are attached. */
int optim_offload_destroy(optim_offload_t* engine);
/* Binds a group to an engine (before its first offloaded step); OPTIM_EINVAL if a state buffer is
 * not pinned host memory or the group does not fit in one slot.  Destroying the group unbinds it. */
int optim_group_attach_offload(optim_group_t* group, optim_offload_t* engine);

/* Layout of a group's host image: total_bytes (the image size), and, if offsets is not NULL,
 * 3 byte offsets per tensor in group order -- residual, m buffer, v buffer, each at a 256-byte
 * boundary, -1 for a buffer the tensor does not have (no residual, or numel 0).  The buffers
 * hold exactly what the group's device buffers would (lmopt.h layouts of each kind); the gaps
 * between them carry nothing.  OPTIM_EINVAL for a group kind that cannot be offloaded. */
int optim_offload_layout(optim_group_t* group, int64_t* offsets, int64_t* total_bytes);
/* Moves the group's states into `image`: caller-owned PINNED host memory of at least
 * optim_offload_layout's total_bytes, valid while the group lives.  Between steps only
 * (synchronises the group's last stream, then copies every residual, m and v buffer named at
 * create into the image, from device or host).  From then on the group never touches those
 * buffers again (the caller may free them); the states live in the image and in a staging slot
 * from optim_offload_prefetch to optim_offload_writeback.  OPTIM_EINVAL: not pinned, too small,
 * or a kind that cannot be offloaded; OPTIM_ESTATE: already attached, or the library's ring
 * must grow while another group's states are on the device. */
int optim_group_attach_host(optim_group_t* group, void* image, size_t bytes);
/* Enqueues on `copy` the copy-in of the group's states into a staging slot (nothing if the group
 * already holds one).  The copy waits (device-side) until the slot's previous write-back is done.
 * copy: a cudaStream_t as void*; NULL = the library's own H2D stream (the engine's, or the
 * library ring's).  A later step of the group waits for the copy on its own stream. */
int optim_offload_prefetch(optim_group_t* group, void* copy);
/* Enqueues on `copy` the copy-out of the group's states after its last step (device-side wait
 * for that step) and releases the slot; the image is valid once `copy` has finished it.  NULL =
 * the library's own D2H stream (waited for by optim_offload_sync(NULL, ...)).  For groups
 * attached with optim_group_attach_host; engine-attached groups write back at the end of every
 * step, and this call does nothing for them.  OPTIM_ESTATE if the group holds no slot. */
int optim_offload_writeback(optim_group_t* group, void* copy);
/* Bounded wait for the copies on the engine's own streams (engine NULL: the library ring of the
 * current device); returns the bytes copied in each direction so far. */
int optim_offload_sync(optim_offload_t* engine, uint64_t* bytes_h2d, uint64_t* bytes_d2h);

/* Profiling hook: when `event` (a cudaEvent_t passed as void*) is not NULL, the next step calls
 * of this group record it on their stream between the pre-pass (gradient max, or the factored
 * statistics passes) and the update kernel, so that a caller can time the two phases with its
 * own events around the call (factored groups of several waves: before the last wave's update
 * kernel, on the stream that wave runs on).  NULL turns it off. */
int optim_group_set_profile_event(optim_group_t* group, void* event);

const char* optim_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LMOPT_H */
