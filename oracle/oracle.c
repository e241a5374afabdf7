/*
 * oracle.c -- plain, slow, single-threaded CPU oracle of the fused optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Arithmetic.  The pages fix fp32 for the update: the master weight is an f32 value that is
 * restored bit-identically from its bf16 upper half and the 16 low bits ("Kahan summation for
 * Adafactor-optimized Flux FFT", sd-scripts PR #2159, first comment), and the printed fused
 * Adafactor step casts grad and weight to float32 before updating ("Fused backward pass" commit,
 * library/adafactor_fused.py, adafactor_step_param).  So every per-element operation below is a
 * single IEEE fp32 operation rounded to nearest-even, in the order written: a*b+c written as
 * fmaf() is one fused rounding (C99 fmaf is exact), everything else rounds per operation and
 * nothing is contracted implicitly (build with -ffp-contract=off).  Means over rows, columns
 * and tensors are summed in double and rounded once to fp32.  Per-step host scalars are
 * computed in double and rounded once.
 *
 * Readings of the pages that this file fixes (each one is listed with its reason in the design
 * notes of the repository):
 *   R1  Kahan split = truncation: hi = upper 16 bits of the f32 pattern, lo = lower 16 bits.
 *   R2  NAdam = Dozat's Nesterov Adam with the momentum schedule mu_t = b1 (1 - 0.5*0.96^(t psi)).
 *   R3  u16 codec for exp_avg: code = 32768 + sgn(m) rint(32767 sqrt(|m|/S)); decode
 *       m = S t|t|, t = (code-32768)/32767.  For exp_avg_sq: code = rint(65535 (v/S)^(1/4));
 *       decode v = S z^4, z = code/65535.  Scale and code step are folded into per-tensor
 *       constants (orc_codec_consts).
 *   R4  Per-tensor scale for step t: S_m = b1 A_m(t-1) + (1-b1) G(t), S_v = b2 A_v(t-1) +
 *       (1-b2) G(t)^2, with A the max over the tensor of the pre-encode moments at t-1 and
 *       G(t) = max |g(t)|.
 *   R5  Tensors of 4096 or fewer elements keep fp32 moments (no codec).
 *   R6  Factored second moment: means of g^2+eps1 over the last dim (rows) and the second-to-last
 *       dim (columns); V^ = R C / mean(R); update clipped by max(1, RMS/clip).
 *   R19 Prodigy's step-size estimate d over the factored step, on a sliced subsample (see the
 *       section of that name).
 *
 * Parity pins (tests/test_oracle_*.py) tie this file to what the pages and mathematics fix:
 * exhaustive split/merge round trip, IEEE bit patterns, exhaustive codec round trip, Adam
 * step-1 = lr sign(g), NAdam step-1 closed form, torch.optim.{Adam,AdamW,NAdam,Adafactor}
 * special cases, rank-1 factored case, zero-gradient and decay-only closed forms, Prodigy's
 * d under a constant gradient (a scalar recurrence) and its independence of the slicing.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <float.h>
#include <stdlib.h>

#define ORC_SMALL_NUMEL 4096

uint32_t orc_sr_bits(uint64_t seed, uint32_t tensor, int64_t step, int64_t i);
static uint16_t sr_bf16(float x, uint32_t r16);

/* ----------------------------------------------------------------------------------------
 * bit helpers
 * -------------------------------------------------------------------------------------- */
static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b_of(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }
static float bf16_to_f32(uint16_t h) { return f_of((uint32_t)h << 16); }

/* ----------------------------------------------------------------------------------------
 * R1: Kahan split / merge.  The bf16 weight is the upper half of the f32 master and the
 * residual is the 16 low bits that bf16 drops, so merge(split(x)) == x for every pattern.
 * -------------------------------------------------------------------------------------- */
void orc_kahan_split(const float* x, uint16_t* hi, uint16_t* lo, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = b_of(x[i]);
        hi[i] = (uint16_t)(b >> 16);
        lo[i] = (uint16_t)(b & 0xFFFFu);
    }
}

void orc_kahan_merge(const uint16_t* hi, const uint16_t* lo, float* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        x[i] = f_of(((uint32_t)hi[i] << 16) | (uint32_t)lo[i]);
}

/* Round-to-nearest-even f32 -> bf16 (the store used when no residual is kept).  Ties go to the
 * even upper half; NaN stays NaN (quiet bit set), infinities stay infinities. */
static uint16_t rne_bf16(float x)
{
    uint32_t b = b_of(x);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0)
        return (uint16_t)((b >> 16) | 0x0040u);
    uint32_t up = b >> 16, rem = b & 0xFFFFu;
    if (rem > 0x8000u || (rem == 0x8000u && (up & 1u)))
        up += 1u;
    return (uint16_t)up;
}

void orc_round_bf16(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = rne_bf16(x[i]);
}

/* ----------------------------------------------------------------------------------------
 * R3: u16 companded codec (sd-scripts PR #2187, second post: both moments are scaled, stored as
 * biased uint16 codes, and pass through a power curve; the constants are not given).
 * Curve: exp_avg code = 32768 + sgn(m) rint(32767 (|m|/S)^(1/2)), exp_avg_sq code =
 * rint(65535 (v/S)^(1/4)).  The code step and the scale are folded into per-tensor constants,
 * computed once per tensor from S:
 *   qm = sqrt(S) * (1/32767)      decode  m = t |t|,  t = (code - 32768) qm
 *   rm = 1 / (qm qm)              encode  k = rint(min(sqrt(|m| rm), 32767))
 *   qv = sqrt(sqrt(S)) * (1/65535) decode v = (z z)(z z), z = code qv
 *   rv = 1 / (qv qv)              encode  k = rint(min(sqrt(sqrt(v) rv), 65535))
 * (rm, rv: 0 when S = 0, at most FLT_MAX otherwise).  Each written operation is one fp32
 * rounding; sqrt is IEEE-correct; rint rounds half to even.
 * -------------------------------------------------------------------------------------- */
typedef struct { float qm, rm, qv, rv; } orc_codec_t;

void orc_codec_consts(float s_m, float s_v, orc_codec_t* c)
{
    c->qm = sqrtf(s_m) * (1.0f / 32767.0f);
    c->rm = (s_m > 0.0f) ? fminf(1.0f / (c->qm * c->qm), FLT_MAX) : 0.0f;
    c->qv = sqrtf(sqrtf(s_v)) * (1.0f / 65535.0f);
    c->rv = (s_v > 0.0f) ? fminf(1.0f / (c->qv * c->qv), FLT_MAX) : 0.0f;
}

uint16_t orc_encode_m(float m, float rm)
{
    float a = fabsf(m) * rm;
    float y = sqrtf(a);
    float k = rintf(fminf(y, 32767.0f));
    uint32_t kk = (uint32_t)k;
    return (uint16_t)(signbit(m) ? 32768u - kk : 32768u + kk);
}

float orc_decode_m(uint16_t c, float qm)
{
    float t = (float)((int32_t)c - 32768) * qm;
    return t * fabsf(t);
}

/* sv is sqrt(v); the update needs that root anyway, so the codec reuses it. */
uint16_t orc_encode_v(float sv, float rv)
{
    float y = sqrtf(sv * rv);
    float k = rintf(fminf(y, 65535.0f));
    return (uint16_t)(uint32_t)k;
}

float orc_decode_v(uint16_t c, float qv)
{
    float z = (float)c * qv;
    float z2 = z * z;
    return z2 * z2;
}

/* Stand-alone pack: S = max over the buffer (|x| for exp_avg, x for exp_avg_sq), then encode. */
void orc_state_pack(const float* x, uint16_t* codes, float* scale, int64_t n, int32_t is_signed)
{
    uint32_t mx = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = b_of(x[i]) & 0x7FFFFFFFu;
        if (b > mx) mx = b;
    }
    float s = f_of(mx);
    *scale = s;
    orc_codec_t c;
    orc_codec_consts(s, s, &c);
    for (int64_t i = 0; i < n; ++i)
        codes[i] = is_signed ? orc_encode_m(x[i], c.rm) : orc_encode_v(sqrtf(x[i]), c.rv);
}

void orc_state_unpack(const uint16_t* codes, float scale, float* x, int64_t n, int32_t is_signed)
{
    orc_codec_t c;
    orc_codec_consts(scale, scale, &c);
    for (int64_t i = 0; i < n; ++i)
        x[i] = is_signed ? orc_decode_m(codes[i], c.qm) : orc_decode_v(codes[i], c.qv);
}

/* ----------------------------------------------------------------------------------------
 * R2: per-step host scalars of Adam / NAdam, double then one rounding to fp32.
 *   Adam:  c_m = 1/(1-b1^t), c_g = 0
 *   NAdam: mu_t = b1 (1 - 0.5*0.96^(t psi)), P_t = P_{t-1} mu_t,
 *          c_g = (1-mu_t)/(1-P_t), c_m = mu_{t+1}/(1 - P_t mu_{t+1})
 *   both:  k2 = 1/sqrt(1-b2^t)
 * The pages name Nesterov momentum, that is NAdamW (sd-scripts PR #2187, first post), without
 * printing a formula; this is Dozat's NAdam with the usual momentum-decay schedule.
 * -------------------------------------------------------------------------------------- */
typedef struct {
    float lr, b1, omb1, b2, omb2, eps, lr_wd, c_m, c_g, k2;
    int32_t decoupled_wd;
} orc_nadam_scalars_t;

void orc_nadam_scalars(int64_t t, float lr, float beta1, float beta2, float eps, float wd,
                       int32_t decoupled_wd, int32_t nesterov, float psi, double* mu_product,
                       orc_nadam_scalars_t* k)
{
    double b1 = beta1, b2 = beta2, td = (double)t;
    k->lr = lr;
    k->b1 = beta1;
    k->omb1 = (float)(1.0 - b1);
    k->b2 = beta2;
    k->omb2 = (float)(1.0 - b2);
    k->eps = eps;
    k->lr_wd = (float)((double)lr * (double)wd);
    k->decoupled_wd = decoupled_wd;
    k->k2 = (float)(1.0 / sqrt(1.0 - pow(b2, td)));
    if (nesterov) {
        double mu = b1 * (1.0 - 0.5 * pow(0.96, td * (double)psi));
        double mu_next = b1 * (1.0 - 0.5 * pow(0.96, (td + 1.0) * (double)psi));
        double prod = *mu_product * mu;
        *mu_product = prod;
        k->c_g = (float)((1.0 - mu) / (1.0 - prod));
        k->c_m = (float)(mu_next / (1.0 - prod * mu_next));
    } else {
        k->c_m = (float)(1.0 / (1.0 - pow(b1, td)));
        k->c_g = 0.0f;
    }
}

/* Per-tensor scale record.  s_m, s_v: scales the stored codes were encoded with (decode slot);
 * a_m, a_v: max |m| and max v of the fp32 moments before encoding, at the last step. */
typedef struct { float s_m, s_v, a_m, a_v; } orc_scale_t;

/* G = max |g| over the tensor, taken on the bf16 magnitude bits (equal to the float max for
 * every non-NaN input; a NaN magnitude compares above infinity, so a NaN gradient makes the
 * tensor's scale NaN and is reported by the non-finite count). */
float orc_grad_absmax(const uint16_t* g, int64_t n)
{
    uint32_t mx = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = g[i] & 0x7FFFu;
        if (b > mx) mx = b;
    }
    return bf16_to_f32((uint16_t)mx);
}

/* ----------------------------------------------------------------------------------------
 * One NAdam(W)/Adam step of one tensor with the Kahan residual and companded states.
 *   hi : bf16 weight bits (in/out);  lo : residual bits (in/out), or NULL for a plain RNE store
 *   m, v : uint16 codes if n > 4096, else fp32 (R5)
 *   g  : bf16 gradient bits
 * Order per element (moments first, then decoupled decay, then the update -- the printed
 * Adafactor step decays the weight before subtracting the update); fma() is one rounding:
 *   w  = merge(hi, lo);  g = f32(g)
 *   m  = fma(b1, m0, (1-b1) g);   v = fma(b2, v0, (1-b2) (g g))
 *   w  = fma(-(lr wd), w, w)                            (decoupled decay only)
 *   sv = sqrt(v);  den = fma(sv, k2, eps);  num = fma(c_m, m, c_g g)
 *   w  = fma(-lr, num / den, w);  (hi, lo) = split(w)
 * The update uses the fp32 moments just computed; quantisation happens only between steps
 * (PR #2187, third post: the compact format holds values between steps and is not computed in).
 * The scale maxima A_m = max |m|, A_v = max v skip NaN (fmax semantics).
 * -------------------------------------------------------------------------------------- */
static float nadam_elem(float w, float gg, float* mm, float* vv, float* sv,
                        const orc_nadam_scalars_t* k)
{
    *mm = fmaf(k->b1, *mm, k->omb1 * gg);
    *vv = fmaf(k->b2, *vv, k->omb2 * (gg * gg));
    if (k->decoupled_wd)
        w = fmaf(-k->lr_wd, w, w);
    *sv = sqrtf(*vv);
    float den = fmaf(*sv, k->k2, k->eps);
    float num = fmaf(k->c_m, *mm, k->c_g * gg);
    return fmaf(-k->lr, num / den, w);
}

/* One step of one tensor whose gradient maximum G is given: the scale is a property of the
 * whole tensor, so a tensor split into slices steps each slice with the maximum over all slices
 * (and with the maxima A_m, A_v over all slices in the scale record).  `small` chooses the fp32
 * moments of tensors of 4096 or fewer elements, decided on the whole tensor. */
void orc_nadam_step_slice(uint16_t* hi, uint16_t* lo, void* m, void* v, const uint16_t* g,
                          int64_t n, int32_t small, float G, orc_scale_t* sc, const orc_nadam_scalars_t* k)
{
    float s_m = 0.0f, s_v = 0.0f;
    orc_codec_t dec, enc;
    if (!small) {
        s_m = fmaf(k->b1, sc->a_m, k->omb1 * G);
        s_v = fmaf(k->b2, sc->a_v, k->omb2 * (G * G));
        orc_codec_consts(sc->s_m, sc->s_v, &dec);
        orc_codec_consts(s_m, s_v, &enc);
    }
    float am = 0.0f, av = 0.0f;
    uint16_t* mc = (uint16_t*)m;
    uint16_t* vc = (uint16_t*)v;
    float* mf = (float*)m;
    float* vf = (float*)v;
    for (int64_t i = 0; i < n; ++i) {
        float w = lo ? f_of(((uint32_t)hi[i] << 16) | lo[i]) : bf16_to_f32(hi[i]);
        float gg = bf16_to_f32(g[i]);
        float mm = small ? mf[i] : orc_decode_m(mc[i], dec.qm);
        float vv = small ? vf[i] : orc_decode_v(vc[i], dec.qv);
        float sv;
        w = nadam_elem(w, gg, &mm, &vv, &sv, k);
        if (lo) {
            uint32_t b = b_of(w);
            hi[i] = (uint16_t)(b >> 16);
            lo[i] = (uint16_t)(b & 0xFFFFu);
        } else {
            hi[i] = rne_bf16(w);
        }
        if (small) {
            mf[i] = mm;
            vf[i] = vv;
        } else {
            mc[i] = orc_encode_m(mm, enc.rm);
            vc[i] = orc_encode_v(sv, enc.rv);
            am = fmaxf(am, fabsf(mm));
            av = fmaxf(av, vv);
        }
    }
    if (!small) {
        sc->s_m = s_m;
        sc->s_v = s_v;
        sc->a_m = am;
        sc->a_v = av;
    }
}

void orc_nadam_step_tensor(uint16_t* hi, uint16_t* lo, void* m, void* v, const uint16_t* g,
                           int64_t n, orc_scale_t* sc, const orc_nadam_scalars_t* k)
{
    int small = n <= ORC_SMALL_NUMEL;
    orc_nadam_step_slice(hi, lo, m, v, g, n, small, small ? 0.0f : orc_grad_absmax(g, n), sc, k);
}

/* ----------------------------------------------------------------------------------------
 * f24 moment storage (sd-scripts PR #2187, third post: f24 keeps the top three bytes of an fp32
 * value, eight mantissa bits more than bf16, and serves as storage only, not for arithmetic).  Reading: the stored value is the f32 pattern truncated to its upper 24 bits
 * (like the Kahan split); decode appends a zero byte.  Layout per moment buffer of n elements:
 * n uint16 words of the upper 16 bits, zero padding up to byte offset 2n rounded up to a
 * multiple of 16, then n bytes of bits 8..15 (storage only: the padding carries no value).  No scale is needed, so no
 * gradient maximum either.  Tensors of 4096 or fewer elements keep fp32 moments as before.
 * -------------------------------------------------------------------------------------- */
static float f24_load(const uint8_t* buf, int64_t n, int64_t i)
{
    const uint16_t* hi = (const uint16_t*)buf;
    const uint8_t* lo = buf + ((2 * n + 15) / 16) * 16;
    return f_of(((uint32_t)hi[i] << 16) | ((uint32_t)lo[i] << 8));
}

static void f24_store(uint8_t* buf, int64_t n, int64_t i, float x)
{
    uint16_t* hi = (uint16_t*)buf;
    uint8_t* lo = buf + ((2 * n + 15) / 16) * 16;
    uint32_t b = b_of(x);
    hi[i] = (uint16_t)(b >> 16);
    lo[i] = (uint8_t)((b >> 8) & 0xFFu);
}

/* sr != 0 (and lo == NULL): the new weight is stochastically rounded (see orc_sr_bits below). */
void orc_nadam_step_tensor_f24(uint16_t* hi, uint16_t* lo, void* m, void* v, const uint16_t* g,
                               int64_t n, const orc_nadam_scalars_t* k, int32_t sr, uint64_t seed,
                               uint32_t tensor, int64_t step)
{
    int small = n <= ORC_SMALL_NUMEL;
    for (int64_t i = 0; i < n; ++i) {
        float w = lo ? f_of(((uint32_t)hi[i] << 16) | lo[i]) : bf16_to_f32(hi[i]);
        float gg = bf16_to_f32(g[i]);
        float mm = small ? ((float*)m)[i] : f24_load((const uint8_t*)m, n, i);
        float vv = small ? ((float*)v)[i] : f24_load((const uint8_t*)v, n, i);
        float sv;
        w = nadam_elem(w, gg, &mm, &vv, &sv, k);
        if (lo) {
            uint32_t b = b_of(w);
            hi[i] = (uint16_t)(b >> 16);
            lo[i] = (uint16_t)(b & 0xFFFFu);
        } else if (sr) {
            hi[i] = sr_bf16(w, orc_sr_bits(seed, tensor, step, i));
        } else {
            hi[i] = rne_bf16(w);
        }
        if (small) {
            ((float*)m)[i] = mm;
            ((float*)v)[i] = vv;
        } else {
            f24_store((uint8_t*)m, n, i, mm);
            f24_store((uint8_t*)v, n, i, vv);
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * Stochastic rounding of the fp32 master to bf16, in place of the Kahan residual ("Kahan summation
 * for Adafactor-optimized Flux FFT", sd-scripts PR #2159, PR description: the value goes to the
 * bf16 neighbour above or below at random, with odds set by how close it is to each).  Reading: add 16 uniform random bits to the f32 pattern and keep
 * the upper half, which rounds the magnitude up with probability (low 16 bits)/65536.
 * Random bits: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011): four 32-bit counter words, two key words, ten rounds; each round forms
 * the two 64-bit products M0*c0 and M1*c2, the new words are (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2),
 * hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)), and the key is bumped by the Weyl constants.  The pages do
 * not name a generator; this one is chosen as a published counter-based generator that both
 * sides can compute independently per element.  Key (seed mod 2^32, seed / 2^32); counter
 * (b mod 2^32, b / 2^32, tensor index, step mod 2^32) with b = i / 8; element i takes 16-bit
 * lane i mod 8 of the 128-bit block (word (i mod 8) / 2, low half for even i).
 * -------------------------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint32_t orc_sr_bits(uint64_t seed, uint32_t tensor, int64_t step, int64_t i)
{
    uint64_t b = (uint64_t)i >> 3;
    uint32_t ctr[4] = {(uint32_t)b, (uint32_t)(b >> 32), tensor, (uint32_t)step};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)}, out[4];
    orc_philox4x32_10(ctr, key, out);
    int lane = (int)(i & 7);
    return (out[lane >> 1] >> (16 * (lane & 1))) & 0xFFFFu;
}

static uint16_t sr_bf16(float x, uint32_t r16)
{
    uint32_t b = b_of(x);
    if ((b & 0x7F800000u) == 0x7F800000u) return (uint16_t)(b >> 16);   /* inf / NaN kept */
    return (uint16_t)((b + r16) >> 16);
}

void orc_stochastic_round(const float* x, uint16_t* out, int64_t n, uint64_t seed, uint32_t tensor, int64_t step)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sr_bf16(x[i], orc_sr_bits(seed, tensor, step, i));
}

/* NAdam/Adam step without a residual, the new fp32 weight stochastically rounded to bf16
 * (u16 or fp32 moments as in orc_nadam_step_tensor). */
void orc_nadam_step_tensor_sr(uint16_t* hi, void* m, void* v, const uint16_t* g, int64_t n,
                              orc_scale_t* sc, const orc_nadam_scalars_t* k, uint64_t seed,
                              uint32_t tensor, int64_t step)
{
    /* the update itself is the no-residual step; only the final store differs */
    int small = n <= ORC_SMALL_NUMEL;
    float s_m = 0.0f, s_v = 0.0f;
    orc_codec_t dec, enc;
    if (!small) {
        float G = orc_grad_absmax(g, n);
        s_m = fmaf(k->b1, sc->a_m, k->omb1 * G);
        s_v = fmaf(k->b2, sc->a_v, k->omb2 * (G * G));
        orc_codec_consts(sc->s_m, sc->s_v, &dec);
        orc_codec_consts(s_m, s_v, &enc);
    }
    float am = 0.0f, av = 0.0f;
    uint16_t* mc = (uint16_t*)m;
    uint16_t* vc = (uint16_t*)v;
    float* mf = (float*)m;
    float* vf = (float*)v;
    for (int64_t i = 0; i < n; ++i) {
        float w = bf16_to_f32(hi[i]);
        float gg = bf16_to_f32(g[i]);
        float mm = small ? mf[i] : orc_decode_m(mc[i], dec.qm);
        float vv = small ? vf[i] : orc_decode_v(vc[i], dec.qv);
        float sv;
        w = nadam_elem(w, gg, &mm, &vv, &sv, k);
        hi[i] = sr_bf16(w, orc_sr_bits(seed, tensor, step, i));
        if (small) {
            mf[i] = mm;
            vf[i] = vv;
        } else {
            mc[i] = orc_encode_m(mm, enc.rm);
            vc[i] = orc_encode_v(sv, enc.rv);
            am = fmaxf(am, fabsf(mm));
            av = fmaxf(av, vv);
        }
    }
    if (!small) {
        sc->s_m = s_m;
        sc->s_v = s_v;
        sc->a_m = am;
        sc->a_v = av;
    }
}

/* ----------------------------------------------------------------------------------------
 * Adan (sd-scripts PR #2187, fourth post: an offloaded Adan, which keeps four states per
 * parameter; Algorithm 1 of the linked paper, arXiv
 * 2208.06677, with its convention that beta weights the new term):
 *   d = g - g_prev
 *   m = (1-b1) m + b1 g;  v = (1-b2) v + b2 d;  n = (1-b3) n + b3 (g + (1-b2) d)^2
 *   w = (w - lr (m + (1-b2) v) / (sqrt(n) + eps)) / (1 + lr wd)
 * Readings: the first step initialises m = g, v = 0, n = g^2 (zero difference), the second sets
 * v = d exactly (the paper's v_1 = g_1 - g_0); states m, v, n fp32 (the pages leave their
 * compression unspecified) and g_prev the previous bf16 gradient.  Per element, fma = one rounding:
 *   m  = fma(omb1, m, b1 g);  v = fma(omb2, v, b2 d);  c = fma(omb2, d, g);  n = fma(omb3, n, b3 (c c))
 *   den = sqrt(n) + eps;  u = fma(omb2, v, m);  w = (w - lr (u / den)) * inv_decay
 * with inv_decay = 1/(1 + lr wd) computed once per step in double.
 * mnv: fp32 planes m, v, n, each P = n rounded up to a multiple of 4 long (the padding is
 * storage only: it keeps every plane 16-byte aligned); gprev: bf16 bits [n].
 * -------------------------------------------------------------------------------------- */
typedef struct {
    float lr, b1, omb1, b2, omb2, b3, omb3, eps, inv_decay;
} orc_adan_scalars_t;

void orc_adan_scalars(float lr, float b1, float b2, float b3, float eps, float wd, orc_adan_scalars_t* k)
{
    k->lr = lr;
    k->b1 = b1;
    k->omb1 = (float)(1.0 - (double)b1);
    k->b2 = b2;
    k->omb2 = (float)(1.0 - (double)b2);
    k->b3 = b3;
    k->omb3 = (float)(1.0 - (double)b3);
    k->eps = eps;
    k->inv_decay = (float)(1.0 / (1.0 + (double)lr * (double)wd));
}

static float adan_elem(float w, float gg, float gp, float* m, float* v, float* nn, int64_t step,
                       const orc_adan_scalars_t* k)
{
    float d = gg - gp;
    if (step == 1) {
        *m = gg;
        *v = 0.0f;
        *nn = gg * gg;
    } else {
        *m = fmaf(k->omb1, *m, k->b1 * gg);
        *v = step == 2 ? d : fmaf(k->omb2, *v, k->b2 * d);
        float c = fmaf(k->omb2, d, gg);
        *nn = fmaf(k->omb3, *nn, k->b3 * (c * c));
    }
    float den = sqrtf(*nn) + k->eps;
    float u = fmaf(k->omb2, *v, *m);
    return (w - k->lr * (u / den)) * k->inv_decay;
}

static void adan_store_w(uint16_t* hi, uint16_t* lo, int64_t i, float w, int32_t sr, uint64_t seed,
                         uint32_t tensor, int64_t step)
{
    if (lo) {
        uint32_t b = b_of(w);
        hi[i] = (uint16_t)(b >> 16);
        lo[i] = (uint16_t)(b & 0xFFFFu);
    } else if (sr) {
        hi[i] = sr_bf16(w, orc_sr_bits(seed, tensor, step, i));
    } else {
        hi[i] = rne_bf16(w);
    }
}

void orc_adan_step_tensor(uint16_t* hi, uint16_t* lo, float* mnv, uint16_t* gprev, const uint16_t* g,
                          int64_t n, int64_t step, const orc_adan_scalars_t* k, int32_t sr, uint64_t seed,
                          uint32_t tensor)
{
    const int64_t P = (n + 3) / 4 * 4;
    float* m = mnv;
    float* v = mnv + P;
    float* nn = mnv + 2 * P;
    for (int64_t i = 0; i < n; ++i) {
        float w = lo ? f_of(((uint32_t)hi[i] << 16) | lo[i]) : bf16_to_f32(hi[i]);
        float mm = m[i], vv = v[i], n2 = nn[i];
        w = adan_elem(w, bf16_to_f32(g[i]), bf16_to_f32(gprev[i]), &mm, &vv, &n2, step, k);
        m[i] = mm;
        v[i] = vv;
        nn[i] = n2;
        gprev[i] = g[i];
        adan_store_w(hi, lo, i, w, sr, seed, tensor, step);
    }
}

/* Adan with its three states stored as f24 (the compact storage the same page describes for the
 * NAdam moments, applied to Adan's m, v and n, whose compression that page leaves open).  Each
 * state is an f24 buffer as above (upper-16-bit plane, zero padding to 16 bytes, byte plane),
 * padded to a multiple of 16 bytes; the three follow each other in `buf`, state j at byte
 * j * F, F = f24 bytes of n rounded up to 16.  Tensors of 4096 or fewer elements keep the fp32
 * planes of orc_adan_step_tensor.  As for the NAdam moments, the update computes on the
 * decoded fp32 states and only the stored values are truncated. */
int64_t orc_adan_f24_stride(int64_t n)
{
    return (((2 * n + 15) / 16) * 16 + n + 15) / 16 * 16;
}

void orc_adan_step_tensor_f24(uint16_t* hi, uint16_t* lo, uint8_t* buf, uint16_t* gprev, const uint16_t* g,
                              int64_t n, int64_t step, const orc_adan_scalars_t* k, int32_t sr, uint64_t seed,
                              uint32_t tensor)
{
    if (n <= ORC_SMALL_NUMEL) {
        orc_adan_step_tensor(hi, lo, (float*)buf, gprev, g, n, step, k, sr, seed, tensor);
        return;
    }
    const int64_t F = orc_adan_f24_stride(n);
    uint8_t* mb = buf;
    uint8_t* vb = buf + F;
    uint8_t* nb = buf + 2 * F;
    for (int64_t i = 0; i < n; ++i) {
        float w = lo ? f_of(((uint32_t)hi[i] << 16) | lo[i]) : bf16_to_f32(hi[i]);
        float mm = f24_load(mb, n, i), vv = f24_load(vb, n, i), n2 = f24_load(nb, n, i);
        w = adan_elem(w, bf16_to_f32(g[i]), bf16_to_f32(gprev[i]), &mm, &vv, &n2, step, k);
        f24_store(mb, n, i, mm);
        f24_store(vb, n, i, vv);
        f24_store(nb, n, i, n2);
        gprev[i] = g[i];
        adan_store_w(hi, lo, i, w, sr, seed, tensor, step);
    }
}

/* Same step with a plain fp32 master weight and fp32 moments (no Kahan split, no codec):
 * the textbook optimizer the Kahan path must reproduce bit for bit given equal moments. */
void orc_nadam_step_fp32(float* w, float* m, float* v, const uint16_t* g, int64_t n,
                         const orc_nadam_scalars_t* k)
{
    for (int64_t i = 0; i < n; ++i) {
        float sv;
        w[i] = nadam_elem(w[i], bf16_to_f32(g[i]), &m[i], &v[i], &sv, k);
    }
}

/* ----------------------------------------------------------------------------------------
 * R6: factored second moment (Adafactor; Prodigy's factored variant), beta1 = 0, no exp_avg.
 * Follows the printed fused Adafactor step ("Fused backward pass" commit,
 * library/adafactor_fused.py, adafactor_step_param) with a fixed learning rate, and the eps2
 * placement of prodigy PR #25 ("more VRAM savings: no first moment and factored second
 * moment", the comment that moves eps2 out of the d^2 scaling).
 *
 * mode 0 (Adafactor): b2t = 1 - t^decay_rate, q = g g + eps1,
 *                     R = b2t R + (1-b2t) mean_j q, C = b2t C + (1-b2t) mean_i q
 * mode 1 (Prodigy):   q = g g, R = b2 R + d^2 (1-b2) mean_j q + eps2, C likewise
 * V^_ij = R_i C_j / mean_i(R);  u_ij = (rsqrt(R_i / mean R) rsqrt(C_j)) g_ij
 * 1-D:   V = b2t V + (1-b2t) q (mode 1: + eps2);  u = rsqrt(V) g
 * mode 1 then takes u = u d: with beta1 = 0 Prodigy's first moment is d g, so the numerator
 * carries d as the second moment carries d^2.
 * then   u = (u / max(1, RMS(u)/clip)) lr_eff;  w = w + w (-wd lr_eff);  w = w - u;  split.
 * lr_eff = lr in mode 0 and d lr in mode 1.
 * -------------------------------------------------------------------------------------- */
typedef struct {
    float b2t, alpha, eps1, eps2, clip, lr_eff, nwdlr;
    int32_t mode;
    float unum;     /* numerator factor: 1 in mode 0, d in mode 1 */
} orc_factored_scalars_t;

void orc_factored_scalars(int64_t t, float lr, float beta2, float decay_rate, float eps1,
                          float eps2, float d, float clip, float wd, int32_t mode,
                          orc_factored_scalars_t* k)
{
    double td = (double)t;
    k->mode = mode;
    k->clip = clip;
    k->eps1 = eps1;
    k->eps2 = eps2;
    if (mode == 0) {
        double beta2t = 1.0 - pow(td, (double)decay_rate);
        k->b2t = (float)beta2t;
        k->alpha = (float)(1.0 - beta2t);
        k->lr_eff = lr;
        k->unum = 1.0f;
    } else {
        k->b2t = beta2;
        k->alpha = (float)((double)d * (double)d * (1.0 - (double)beta2));
        k->lr_eff = (float)((double)d * (double)lr);
        k->unum = d;
    }
    k->nwdlr = (float)(-(double)wd * (double)k->lr_eff);
}

static float rsqrt_rn(float x) { return 1.0f / sqrtf(x); }

/* Update of the weight given the final (unscaled) update u and the clip divisor. */
static void apply_update(uint16_t* hi, uint16_t* lo, int64_t i, float u, float den,
                         const orc_factored_scalars_t* k)
{
    float w = lo ? f_of(((uint32_t)hi[i] << 16) | lo[i]) : bf16_to_f32(hi[i]);
    float uu = (u / den) * k->lr_eff;
    if (k->nwdlr != 0.0f)
        w = w + w * k->nwdlr;
    w = w - uu;
    if (lo) {
        uint32_t b = b_of(w);
        hi[i] = (uint16_t)(b >> 16);
        lo[i] = (uint16_t)(b & 0xFFFFu);
    } else {
        hi[i] = rne_bf16(w);
    }
}

/* max(1, RMS/clip) as the listing's clamp(min=1) computes it: a NaN RMS (an undefined update)
 * stays NaN and makes the whole update NaN, rather than being replaced by 1. */
static float clip_divisor(double ss, int64_t n, float clip)
{
    float ss32 = (float)ss;
    float ms = ss32 / (float)n;
    float rms = sqrtf(ms);
    float r = rms / clip;
    return (r < 1.0f) ? 1.0f : r;
}

/* Factored tensor viewed as B matrices of R rows x C columns (the last two dims), row-major.
 * row[B*R], col[B*C] fp32 state (in/out).  Returns the clip divisor used (for tests). */
float orc_factored_step_tensor(uint16_t* hi, uint16_t* lo, const uint16_t* g, int64_t B,
                               int64_t R, int64_t C, float* row, float* col,
                               const orc_factored_scalars_t* k)
{
    int64_t n = B * R * C;
    /* A tensor without elements has no gradient: nothing is updated, its state included (a mean
     * over zero rows or columns has no value). */
    if (n == 0) return 1.0f;
    /* 1. EMA of row and column means of q */
    for (int64_t b = 0; b < B; ++b) {
        const uint16_t* gb = g + b * R * C;
        for (int64_t i = 0; i < R; ++i) {
            double s = 0.0;
            for (int64_t j = 0; j < C; ++j) {
                float gg = bf16_to_f32(gb[i * C + j]);
                float q = k->mode == 0 ? gg * gg + k->eps1 : gg * gg;
                s += (double)q;
            }
            float r = (float)(s / (double)C);
            float nr = k->b2t * row[b * R + i] + k->alpha * r;
            if (k->mode == 1) nr = nr + k->eps2;
            row[b * R + i] = nr;
        }
        for (int64_t j = 0; j < C; ++j) {
            double s = 0.0;
            for (int64_t i = 0; i < R; ++i) {
                float gg = bf16_to_f32(gb[i * C + j]);
                float q = k->mode == 0 ? gg * gg + k->eps1 : gg * gg;
                s += (double)q;
            }
            float c = (float)(s / (double)R);
            float nc = k->b2t * col[b * C + j] + k->alpha * c;
            if (k->mode == 1) nc = nc + k->eps2;
            col[b * C + j] = nc;
        }
    }
    /* 2. u = rsqrt(R_i / mean R) rsqrt(C_j) g and its sum of squares */
    double ss = 0.0;
    for (int64_t b = 0; b < B; ++b) {
        double rs = 0.0;
        for (int64_t i = 0; i < R; ++i) rs += (double)row[b * R + i];
        float rbar = (float)(rs / (double)R);
        for (int64_t i = 0; i < R; ++i) {
            float rr = rsqrt_rn(row[b * R + i] / rbar);
            for (int64_t j = 0; j < C; ++j) {
                float cc = rsqrt_rn(col[b * C + j]);
                float u = (rr * cc) * bf16_to_f32(g[(b * R + i) * C + j]);
                if (k->mode == 1) u = u * k->unum;
                ss += (double)u * (double)u;
            }
        }
    }
    float den = clip_divisor(ss, n, k->clip);
    /* 3. clip, lr, decay, subtract, split */
    for (int64_t b = 0; b < B; ++b) {
        double rs = 0.0;
        for (int64_t i = 0; i < R; ++i) rs += (double)row[b * R + i];
        float rbar = (float)(rs / (double)R);
        for (int64_t i = 0; i < R; ++i) {
            float rr = rsqrt_rn(row[b * R + i] / rbar);
            for (int64_t j = 0; j < C; ++j) {
                float cc = rsqrt_rn(col[b * C + j]);
                int64_t e = (b * R + i) * C + j;
                float u = (rr * cc) * bf16_to_f32(g[e]);
                if (k->mode == 1) u = u * k->unum;
                apply_update(hi, lo, e, u, den, k);
            }
        }
    }
    return den;
}

/* Non-factored (1-D) tensor: full fp32 second moment V[n] (in/out). */
float orc_factored_step_vector(uint16_t* hi, uint16_t* lo, const uint16_t* g, int64_t n,
                               float* V, const orc_factored_scalars_t* k)
{
    if (n == 0) return 1.0f;   /* no elements: nothing to update (as for matrices) */
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        float gg = bf16_to_f32(g[i]);
        float q = k->mode == 0 ? gg * gg + k->eps1 : gg * gg;
        float nv = k->b2t * V[i] + k->alpha * q;
        if (k->mode == 1) nv = nv + k->eps2;
        V[i] = nv;
        float u = rsqrt_rn(nv) * gg;
        if (k->mode == 1) u = u * k->unum;
        ss += (double)u * (double)u;
    }
    float den = clip_divisor(ss, n, k->clip);
    for (int64_t i = 0; i < n; ++i) {
        float u = rsqrt_rn(V[i]) * bf16_to_f32(g[i]);
        if (k->mode == 1) u = u * k->unum;
        apply_update(hi, lo, i, u, den, k);
    }
    return den;
}

/* ----------------------------------------------------------------------------------------
 * R19: Prodigy's estimate of the step size d on top of the factored step (mode 1).  The pages
 * discuss it (prodigy PR #25: d0, the numerator built from p - p0, "s, which is the denominator
 * in the calculation of d_hat", the EMAs scaled by d) but print no formula; this follows the
 * Adam form of Prodigy in the paper the PR belongs to (Mishchenko, Defazio, "Prodigy: An
 * Expeditiously Adaptive Parameter-Free Learner", 2023), with beta1 = 0 and the factored second
 * moment above.  Over every tensor of every group that shares d, at step k with d_k:
 *     r   = beta3 r + lr d_k^2 sum_e g_e (p0_e - x_e)        (x: the master before the step)
 *     s_e = beta3 s_e + lr d_k^2 g_e
 *     d_{k+1} = max(d_k, r / sum_e |s_e|)                     (d unchanged while sum |s| = 0)
 * (the paper's factor 1 - beta3 on both increments cancels in the quotient and is left out).
 * The statistics are kept on a subsample ("sliced", prodigy PR #22, named by PR #25): of each
 * tensor's flat elements, the 64-element blocks whose block index is a multiple of slice_p
 * (slice_p = 1: every element; a block of 64 bf16 values is one 128-byte line).  p0 and s hold
 * the sampled elements in order, 64 per sampled block, zero where a block runs past the
 * tensor's end.  A step's d is the fp32 value of d_k;
 * lr d_k^2 is formed in double from it, rounded to fp32 for s.
 * -------------------------------------------------------------------------------------- */
int64_t orc_prodigy_slice_len(int64_t n, int32_t slice_p)
{
    int64_t blocks = (n + 63) / 64;
    return 64 * ((blocks + slice_p - 1) / slice_p);
}

static float master_of(const uint16_t* hi, const uint16_t* lo, int64_t e)
{
    return lo ? f_of(((uint32_t)hi[e] << 16) | lo[e]) : bf16_to_f32(hi[e]);
}

/* Flat element of sampled entry j. */
static int64_t sampled_element(int64_t j, int32_t slice_p)
{
    return (j / 64) * (int64_t)slice_p * 64 + (j % 64);
}

void orc_prodigy_snapshot(const uint16_t* hi, const uint16_t* lo, int64_t n, int32_t slice_p, float* p0, float* s)
{
    int64_t len = orc_prodigy_slice_len(n, slice_p);
    for (int64_t j = 0; j < len; ++j) {
        int64_t e = sampled_element(j, slice_p);
        p0[j] = e < n ? master_of(hi, lo, e) : 0.0f;
        s[j] = 0.0f;
    }
}

/* One tensor's share of a step: updates s and adds sum g (p0 - x) to *dot and sum |s| to *l1.
 * cs = fl32(lr d_k^2). */
void orc_prodigy_tensor_stats(const uint16_t* hi, const uint16_t* lo, const uint16_t* g, int64_t n,
                              int32_t slice_p, const float* p0, float* s, float beta3, float cs,
                              double* dot, double* l1)
{
    int64_t len = orc_prodigy_slice_len(n, slice_p);
    for (int64_t j = 0; j < len; ++j) {
        int64_t e = sampled_element(j, slice_p);
        if (e >= n) continue;
        float x = master_of(hi, lo, e);
        float gg = bf16_to_f32(g[e]);
        float diff = p0[j] - x;
        *dot += (double)(gg * diff);
        float sn = beta3 * s[j] + cs * gg;
        s[j] = sn;
        *l1 += (double)fabsf(sn);
    }
}

/* End of a step over all groups: cdot = sum over groups of (lr_g d_k^2) dot_g, in double. */
void orc_prodigy_end_step(double* d, double* r, double beta3, double cdot, double l1)
{
    *r = beta3 * *r + cdot;
    if (l1 > 0.0) {
        double dhat = *r / l1;
        if (dhat > *d) *d = dhat;
    }
}

/* ----------------------------------------------------------------------------------------
 * Timing driver: one NAdam group step spread over the host's threads.  It is not a second
 * definition of the step: every element is updated by orc_nadam_step_slice, unchanged, on a
 * contiguous slice of its tensor; only the per-tensor maxima are combined across slices
 * (max over the slices of max |g|, and of A_m and A_v, which the step takes with fmax, so the
 * result does not depend on how a tensor is cut).  The results are therefore bit-identical to
 * orc_nadam_step_tensor on every tensor (checked by a test).  Built with OpenMP when the
 * compiler has it (the same source, a second library); otherwise it runs on one thread.
 * ptrs[5*i .. 5*i+4] = hi, lo (or NULL), m, v, g of tensor i; n[i] its element count.
 * -------------------------------------------------------------------------------------- */
#ifdef _OPENMP
#include <omp.h>
#endif

int32_t orc_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

#define ORC_SLICE (1 << 20)

void orc_nadam_group_step_mt(int32_t n_tensors, void* const* ptrs, const int64_t* n, orc_scale_t* sc,
                             const orc_nadam_scalars_t* k)
{
    /* work items: (tensor, first element) for every ORC_SLICE elements of every tensor; tensors of
     * 4096 or fewer elements (fp32 moments, no scale) are one item */
    int64_t n_items = 0;
    for (int32_t i = 0; i < n_tensors; ++i)
        n_items += n[i] <= 0 ? 0 : (n[i] + ORC_SLICE - 1) / ORC_SLICE;
    int32_t* it_t = (int32_t*)malloc((size_t)(n_items > 0 ? n_items : 1) * sizeof(int32_t));
    int64_t* it_a = (int64_t*)malloc((size_t)(n_items > 0 ? n_items : 1) * sizeof(int64_t));
    float* part_g = (float*)malloc((size_t)(n_items > 0 ? n_items : 1) * sizeof(float));
    orc_scale_t* part_s = (orc_scale_t*)malloc((size_t)(n_items > 0 ? n_items : 1) * sizeof(orc_scale_t));
    float* tensor_g = (float*)calloc((size_t)(n_tensors > 0 ? n_tensors : 1), sizeof(float));
    int64_t q = 0;
    for (int32_t i = 0; i < n_tensors; ++i)
        for (int64_t a = 0; a < n[i]; a += ORC_SLICE) {
            it_t[q] = i;
            it_a[q] = a;
            ++q;
        }
    /* 1: max |g| of each slice, then of each tensor (exact: a max of bf16 magnitudes) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_items; ++j) {
        int32_t i = it_t[j];
        int64_t a = it_a[j], len = n[i] - a < ORC_SLICE ? n[i] - a : ORC_SLICE;
        part_g[j] = orc_grad_absmax((const uint16_t*)ptrs[5 * i + 4] + a, len);
    }
    for (int64_t j = 0; j < n_items; ++j)
        if (part_g[j] > tensor_g[it_t[j]]) tensor_g[it_t[j]] = part_g[j];
    /* 2: every slice steps with its tensor's G and the tensor's scale record as it was */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < n_items; ++j) {
        int32_t i = it_t[j];
        int64_t a = it_a[j], len = n[i] - a < ORC_SLICE ? n[i] - a : ORC_SLICE;
        int small = n[i] <= ORC_SMALL_NUMEL;
        size_t ms = small ? 4 : 2;
        uint16_t* lo = (uint16_t*)ptrs[5 * i + 1];
        part_s[j] = sc[i];
        orc_nadam_step_slice((uint16_t*)ptrs[5 * i] + a, lo ? lo + a : NULL, (char*)ptrs[5 * i + 2] + ms * (size_t)a,
                             (char*)ptrs[5 * i + 3] + ms * (size_t)a, (const uint16_t*)ptrs[5 * i + 4] + a, len,
                             small, small ? 0.0f : tensor_g[i], &part_s[j], k);
    }
    /* 3: the new record: S from any slice (all equal), A the max over the slices */
    for (int64_t j = 0; j < n_items; ++j) {          /* items are in tensor order, slice 0 first */
        int32_t i = it_t[j];
        if (n[i] <= ORC_SMALL_NUMEL) continue;
        if (it_a[j] == 0) {
            sc[i] = part_s[j];
        } else {
            sc[i].a_m = fmaxf(sc[i].a_m, part_s[j].a_m);
            sc[i].a_v = fmaxf(sc[i].a_v, part_s[j].a_v);
        }
    }
    free(it_t);
    free(it_a);
    free(part_g);
    free(part_s);
    free(tensor_g);
}
