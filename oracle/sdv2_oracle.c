/*
 * Oracle for the streaming causal-video chunk-attention path: plain, slow, CPU-only C.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU-baseline leg
 * may load this file's library.  It shares no code, header, table or constant with the CUDA
 * library: everything here is written from the definitions below.
 *
 * Sources (web pages; the pages give prose only, no equations or listings):
 *  - "Accelerating Video Generation Inference with Sequential-Parallel 3D Positional Encoding
 *    Using a Global Time Index" (gist.science summary), technical summary section 2 (나,
 *    Causal-RoPE SP): positions are computed locally from each block's start-frame index
 *    (global time index); section 2 (다): cos/sin frequencies are precomputed into contiguous
 *    tensors.
 *  - "StreamDiffusionV2" (xllm-io review), section 三 (Sink Token guided rolling KV cache):
 *    sink = KV of the initial frames kept as a global anchor, rolling KV cache = fixed-size
 *    sliding window, RoPE refresh = periodic reset of the positional offset; section 二 table
 *    (motion-aware noise scheduling): L2 motion estimate between adjacent frames.
 *  - The textbook operations those pages name: rotary position embedding over (t, h, w) and
 *    scaled dot-product softmax attention.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - 3D RoPE: head dims split into consecutive t, h, w segments; inside a segment of d_a dims
 *    the pair (2j, 2j+1) turns by angle pos * base^(-2j/d_a); rotation by +angle:
 *    (x, y) -> (x cos - y sin, x sin + y cos).  V is not rotated.
 *  - Rounding of the bf16 path ("spec"): cos and sin are evaluated in fp64 by libm and rounded
 *    once to fp32; each output is bf16_rne(fmaf(x, c, -fp32(y*s))) for the even element and
 *    bf16_rne(fmaf(x, s, fp32(y*c))) for the odd element.
 *  - Attention: softmax(q k^T * scale) v over every retained key, no mask, fp64 throughout.
 *  - Motion: sum over pixels and channels of the squared uint8 difference of adjacent frames,
 *    exact in 64-bit integers.
 *
 * Floating point: compiled with -ffp-contract=off so that no fused multiply-add appears
 * except where fmaf() is written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------------ */
/* bf16 conversions                                                                           */
/* ------------------------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round-to-nearest-even from fp32 to bf16 by integer arithmetic on the bit pattern: add
 * 0x7FFF plus the lowest kept bit, then drop the low 16 bits.  NaN stays NaN (quiet bit set). */
uint16_t orc_f32_to_bf16_rne(float x)
{
    uint32_t u = f32_bits(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* A second, independent formulation of the same rounding, used only to pin the first one:
 * take the two bf16 values that bracket |x| (truncation and the next code up), measure both
 * distances exactly in fp64, pick the nearer, and on a tie the one whose last mantissa bit is
 * zero.  The code above 0x7F7F is treated as the value 2^128 so that the overflow threshold is
 * the IEEE one (max finite + half an ulp).  Returns 0x7FC0 for NaN. */
uint16_t orc_f32_to_bf16_ref(float x)
{
    if (isnan(x)) return 0x7FC0u;
    uint32_t u = f32_bits(x);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag == 0x7F800000u) return (uint16_t)((sign | mag) >> 16);  /* +-inf */
    uint32_t lo = mag & 0xFFFF0000u;
    uint32_t hi = lo + 0x10000u;
    double ax = fabs((double)x);
    double vlo = (double)bits_f32(lo);
    double vhi = (hi == 0x7F800000u) ? ldexp(1.0, 128) : (double)bits_f32(hi);
    double dlo = ax - vlo, dhi = vhi - ax;
    uint32_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = (((lo >> 16) & 1u) == 0) ? lo : hi;
    return (uint16_t)((sign | pick) >> 16);
}

/* Number of fp32 bit patterns in [lo, hi) (hi <= 2^32) on which the two conversions disagree
 * (for NaN inputs both must give a NaN). */
int64_t orc_bf16_mismatches(uint64_t lo, uint64_t hi)
{
    int64_t bad = 0;
#pragma omp parallel for reduction(+ : bad) schedule(static)
    for (int64_t i = (int64_t)lo; i < (int64_t)hi; ++i) {
        float x = bits_f32((uint32_t)i);
        uint16_t a = orc_f32_to_bf16_rne(x);
        uint16_t b = orc_f32_to_bf16_ref(x);
        if (isnan(x)) {
            if (!isnan(orc_bf16_to_f32(a)) || !isnan(orc_bf16_to_f32(b))) ++bad;
        } else if (a != b) {
            ++bad;
        }
    }
    return bad;
}

void orc_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* 3D rotary position embedding                                                                */
/* ------------------------------------------------------------------------------------------ */

/* Frequency of pair j in an axis segment of d_axis dims: base^(-2j/d_axis). */
double orc_rope_omega(int j, int d_axis, double base)
{
    return pow(base, -(double)(2 * j) / (double)d_axis);
}

/* The fp32 cos and sin that the bf16 path uses for position pos, pair j of an axis of d_axis
 * dims: the angle pos*omega in fp64, cos/sin in fp64 (libm), each rounded once to fp32. */
void orc_rope_cos_sin_f32(int64_t pos, int j, int d_axis, double base, float* c, float* s)
{
    double theta = (double)pos * orc_rope_omega(j, d_axis, base);
    *c = (float)cos(theta);
    *s = (float)sin(theta);
}

/* Rotate one head vector of D = dt+dh+dw bf16 values at position (tp, hp, wp): the bf16 path
 * with the rounding spelled out in the file header.  x and y may not alias. */
static void rope_spec_head(const uint16_t* x, uint16_t* y, int dt, int dh, int dw, double base,
                           int64_t tp, int64_t hp, int64_t wp)
{
    const int dims[3] = {dt, dh, dw};
    const int64_t pos[3] = {tp, hp, wp};
    int off = 0;
    for (int a = 0; a < 3; ++a) {
        for (int j = 0; j < dims[a] / 2; ++j) {
            float c, s;
            orc_rope_cos_sin_f32(pos[a], j, dims[a], base, &c, &s);
            float xe = orc_bf16_to_f32(x[off + 2 * j]);
            float xo = orc_bf16_to_f32(x[off + 2 * j + 1]);
            float ys = xo * s;   /* one fp32 rounding */
            float yc = xo * c;   /* one fp32 rounding */
            y[off + 2 * j] = orc_f32_to_bf16_rne(fmaf(xe, c, -ys));
            y[off + 2 * j + 1] = orc_f32_to_bf16_rne(fmaf(xe, s, yc));
        }
        off += dims[a];
    }
}

/* Rotate n head vectors x[n][D] (bf16) whose positions are tpos[n], hpos[n], wpos[n]. */
void orc_rope_spec(const uint16_t* x, uint16_t* y, int64_t n, int dt, int dh, int dw, double base,
                   const int64_t* tpos, const int64_t* hpos, const int64_t* wpos)
{
    const int D = dt + dh + dw;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        rope_spec_head(x + i * D, y + i * D, dt, dh, dw, base, tpos[i], hpos[i], wpos[i]);
}

/* The same rotation in fp64 with no rounding (real-valued positions allowed). */
void orc_rope_ideal(const double* x, double* y, int64_t n, int dt, int dh, int dw, double base,
                    const double* tpos, const double* hpos, const double* wpos)
{
    const int D = dt + dh + dw;
    const int dims[3] = {dt, dh, dw};
    for (int64_t i = 0; i < n; ++i) {
        const double pos[3] = {tpos[i], hpos[i], wpos[i]};
        int off = 0;
        for (int a = 0; a < 3; ++a) {
            for (int j = 0; j < dims[a] / 2; ++j) {
                double th = pos[a] * orc_rope_omega(j, dims[a], base);
                double c = cos(th), s = sin(th);
                double xe = x[i * D + off + 2 * j], xo = x[i * D + off + 2 * j + 1];
                y[i * D + off + 2 * j] = xe * c - xo * s;
                y[i * D + off + 2 * j + 1] = xe * s + xo * c;
            }
            off += dims[a];
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Softmax attention, fp64                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* p = softmax(s) over n scores, fp64 (max subtracted for range only). Returns log-sum-exp. */
double orc_softmax(const double* s, int64_t n, double* p)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) { p[j] = exp(s[j] - m); z += p[j]; }
    for (int64_t j = 0; j < n; ++j) p[j] /= z;
    return m + log(z);
}

/* out[r][:] = sum_j softmax_j(scale * <q_r, k_j>) v_j for nq query rows against nkv keys.
 * q: [nq][D], k and v: [nkv][D], all fp64; out: [nq][D] fp64; lse (nullable): [nq]. */
void orc_attention_f64(const double* q, int64_t nq, const double* k, const double* v, int64_t nkv,
                       int D, double scale, double* out, double* lse)
{
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nkv * sizeof(double));
        double* p = (double*)malloc((size_t)nkv * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nq; ++r) {
            const double* qr = q + r * D;
            for (int64_t j = 0; j < nkv; ++j) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qr[d] * k[j * D + d];
                s[j] = scale * acc;
            }
            double l = orc_softmax(s, nkv, p);
            if (lse) lse[r] = l;
            for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
            for (int64_t j = 0; j < nkv; ++j)
                for (int d = 0; d < D; ++d) out[r * D + d] += p[j] * v[j * D + d];
        }
        free(s);
        free(p);
    }
}

/* The same with bf16 inputs (widened exactly to fp64).  q rows are taken at row indices
 * rows[0..nq) of q_all (so that a sample of rows can be checked at full key length). */
void orc_attention_bf16(const uint16_t* q_all, const int64_t* rows, int64_t nq, const uint16_t* k,
                        const uint16_t* v, int64_t nkv, int D, double scale, double* out, double* lse)
{
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)nkv * sizeof(double));
        double* p = (double*)malloc((size_t)nkv * sizeof(double));
        double* qr = (double*)malloc((size_t)D * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nq; ++r) {
            const uint16_t* qb = q_all + rows[r] * D;
            for (int d = 0; d < D; ++d) qr[d] = (double)orc_bf16_to_f32(qb[d]);
            for (int64_t j = 0; j < nkv; ++j) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qr[d] * (double)orc_bf16_to_f32(k[j * D + d]);
                s[j] = scale * acc;
            }
            double l = orc_softmax(s, nkv, p);
            if (lse) lse[r] = l;
            for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
            for (int64_t j = 0; j < nkv; ++j)
                for (int d = 0; d < D; ++d)
                    out[r * D + d] += p[j] * (double)orc_bf16_to_f32(v[j * D + d]);
        }
        free(s);
        free(p);
        free(qr);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Motion: squared L2 distance of adjacent uint8 frames                                        */
/* ------------------------------------------------------------------------------------------ */

/* sum_i (a[i] - b[i])^2, exact. */
uint64_t orc_ssd_u8(const uint8_t* a, const uint8_t* b, int64_t n)
{
    uint64_t acc = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t d = (int64_t)a[i] - (int64_t)b[i];
        acc += (uint64_t)(d * d);
    }
    return acc;
}

/* frames: [nb][T+1][npix] uint8; ssd: [nb][T]; ssd[b][t] compares frame t+1 with frame t. */
void orc_motion_ssd(const uint8_t* frames, int64_t nb, int64_t T, int64_t npix, uint64_t* ssd)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < nb; ++b)
        for (int64_t t = 0; t < T; ++t) {
            const uint8_t* f0 = frames + (b * (T + 1) + t) * npix;
            ssd[b * T + t] = orc_ssd_u8(f0 + npix, f0, npix);
        }
}

/* ------------------------------------------------------------------------------------------ */
/* Motion-aware noise controller (a declared map; the pages give no formula)                    */
/* ------------------------------------------------------------------------------------------ */

/* rate[b][t] from m[b][t]: u = clamp((m - m_lo)/(m_hi - m_lo), 0, 1), flipped when
 * more_noise_when_fast == 0; r = fmaf(out_hi - out_lo, u, out_lo); the smoothed value is r for a
 * stream's first frame (state < 0) and fmaf(ema, s - r, r) afterwards.  fp32, one rounding per
 * operation as written.  state (nullable) carries s across calls. */
void orc_noise(const float* m, int64_t nb, int64_t T, float m_lo, float m_hi, float out_lo, float out_hi,
               float ema, int more_noise_when_fast, float* state, float* rate)
{
    for (int64_t b = 0; b < nb; ++b) {
        float s = state ? state[b] : -1.0f;
        for (int64_t t = 0; t < T; ++t) {
            float u = (m[b * T + t] - m_lo) / (m_hi - m_lo);
            if (u < 0.0f) u = 0.0f;
            if (u > 1.0f) u = 1.0f;
            if (!more_noise_when_fast) u = 1.0f - u;
            const float r = fmaf(out_hi - out_lo, u, out_lo);
            s = (s < 0.0f) ? r : fmaf(ema, s - r, r);
            rate[b * T + t] = s;
        }
        if (state) state[b] = s;
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
