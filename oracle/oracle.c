/*
 * oracle.c -- plain, slow, scalar CPU oracle for the packed-state AdamW update.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU
 * baseline leg of bench.py are the only code that may load this library.  The
 * product path (libpackedadam.so and its Python binding) never calls it, and
 * the two share no source: no header, table, helper or constant.
 *
 * What it follows (page title, then section):
 *   [PAR] "Packed AdamW Reference" README, v1.0.0, "The canonical format": one
 *         uint32 word per FP32 parameter, low 16 bits a signed finite E4M11
 *         first moment, high 16 bits an unsigned finite E4M12 uncorrected RMS,
 *         no stochastic rounding; the paragraph that follows it: gradients,
 *         bias correction, weight decay and the update stay FP32, the new
 *         moments are used in FP32 and packed afterwards.  The same page names
 *         the FP32 and packed FP16-first/FP16-RMS comparison modes.
 *   [PAC] "Packed AdamW / Reference / v1.0.0" code page, "Release scope":
 *         decode the prior state, square the RMS to get the prior second
 *         moment, compute the next moments and the update in FP32, only then
 *         store the next moment and RMS; formats do not convert themselves at
 *         the finite bound.
 *   [TA]  "TurboAdam" README (turboadam 0.2.0), "The AdamW update remains
 *         AdamW": the AdamW recurrences with decoupled weight decay.
 *   [KB]  KBench task "quantized-optimizer-state", reference.py: the function
 *         quantized_adamw_step (the FP32 operation order, 8-bit blockwise
 *         state, BF16 parameter output) and _requantise (per-2048-block
 *         absmax, nearest entry of an ascending 256-point map via midpoints).
 *
 * Readings taken where the pages are silent (the README's format document is
 * not among the pages):
 *   R1  E4 lanes are IEEE-style with no Inf/NaN codes: E4M11 code =
 *       s<<15 | e<<11 | f, E4M12 code = e<<12 | f; e >= 1 decodes to
 *       2^(e-B) * (1 + f/2^M), e == 0 to 2^(1-B) * f/2^M.
 *   R2  Exponent bias B = 15 for both lanes (E4M11 max 2 - 2^-11, E4M12 max
 *       2 - 2^-12).
 *   R3  Encoding is round to nearest, ties to the even code.
 *   R4  Values at or beyond the largest finite magnitude, and +-Inf, encode to
 *       the signed largest magnitude (saturation).
 *   R5  The sign of zero is kept on the signed lane: -0 and negative values
 *       that round to zero encode to 0x8000, which decodes to -0.0.
 *   R6  NaN encodes to +0 on every lane; the step counts it as non-finite.
 *   R7  The RMS lane is unsigned: negative inputs (and -0) encode to 0.
 *   R8  m' and sqrt(v') are rounded to FP32 first, then to the 16-bit lane.
 *   R9  FP16 lanes are IEEE binary16, round to nearest even, subnormals kept,
 *       saturating at +-65504 instead of overflowing to Inf; NaN -> +0.
 *   R10 Hyperparameter scalars are formed in double and rounded once to FP32;
 *       the per-element update uses the operation order of
 *       quantized_adamw_step, one rounding per operation, no contraction.
 *   R11 Blockwise: n need not be a multiple of 2048; the last block covers the
 *       remaining elements and its absmax is taken over them only.  A NaN in a
 *       block makes its absmax NaN; a NaN normalised value gets code 0 (no
 *       midpoint compares below NaN).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * Every float operation below is one IEEE binary32 operation rounded to
 * nearest even; with contraction off, each source line rounds once.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define E4_BIAS 15

/* ---------------------------------------------------------------------------
 * Decoded value tables.  Each holds the magnitudes of one lane, indexed by the
 * magnitude code, built from the lane's definition (R1, R2, R9).  Encoding is
 * a search for the nearest entry (R3), so the encoder never manipulates bits.
 * ------------------------------------------------------------------------- */
static float e4m11_mag[1u << 15]; /* 4 exponent bits, 11 mantissa bits       */
static float e4m12_mag[1u << 16]; /* 4 exponent bits, 12 mantissa bits       */
static float fp16_mag[31u << 10]; /* binary16 finite magnitudes: e = 0 .. 30 */

/* Value of an IEEE-style magnitude with exponent field e and fraction f of
 * mbits bits: subnormal when e == 0.  ldexp on small integers is exact. */
static double ieee_style_value(uint32_t e, uint32_t f, int mbits, int bias)
{
    if (e == 0)
        return ldexp((double)f, 1 - bias - mbits);
    return ldexp((double)((1u << mbits) + f), (int)e - bias - mbits);
}

__attribute__((constructor)) static void build_tables(void)
{
    for (uint32_t c = 0; c < (1u << 15); ++c)
        e4m11_mag[c] = (float)ieee_style_value(c >> 11, c & 0x7FFu, 11, E4_BIAS);
    for (uint32_t c = 0; c < (1u << 16); ++c)
        e4m12_mag[c] = (float)ieee_style_value(c >> 12, c & 0xFFFu, 12, E4_BIAS);
    for (uint32_t c = 0; c < (31u << 10); ++c)
        fp16_mag[c] = (float)ieee_style_value(c >> 10, c & 0x3FFu, 10, 15);
}

/* Index of the table entry nearest to ax (ax >= 0, not NaN), ties to the even
 * index; at or beyond the last entry, the last entry (R3, R4).  The table is
 * ascending (a property the tests check over every code). */
static uint32_t nearest_code(const float *t, uint32_t count, float ax)
{
    if (ax >= t[count - 1])
        return count - 1;
    uint32_t lo = 0, hi = count - 1; /* t[lo] <= ax < t[hi] */
    while (hi - lo > 1) {
        uint32_t mid = lo + (hi - lo) / 2;
        if (t[mid] <= ax)
            lo = mid;
        else
            hi = mid;
    }
    double below = (double)ax - (double)t[lo];
    double above = (double)t[hi] - (double)ax;
    if (below < above)
        return lo;
    if (above < below)
        return hi;
    return (lo % 2u == 0u) ? lo : hi;
}

/* ---- E4M11, signed first-moment lane ([PAR], [PAC]; R1-R6, R8) ---------- */
float oracle_e4m11_decode(uint16_t code)
{
    float mag = e4m11_mag[code & 0x7FFFu];
    return (code & 0x8000u) ? -mag : mag;
}

uint16_t oracle_e4m11_encode(float x)
{
    if (isnan(x))
        return 0;
    uint32_t mag = nearest_code(e4m11_mag, 1u << 15, fabsf(x));
    return (uint16_t)((signbit(x) ? 0x8000u : 0u) | mag);
}

/* ---- E4M12, unsigned uncorrected-RMS lane ([PAR], [PAC]; R1-R4, R6-R8) -- */
float oracle_e4m12_decode(uint16_t code) { return e4m12_mag[code]; }

uint16_t oracle_e4m12_encode(float x)
{
    if (isnan(x) || signbit(x))
        return 0;
    return (uint16_t)nearest_code(e4m12_mag, 1u << 16, x);
}

/* ---- binary16 lanes of the FP16-first/FP16-RMS mode ([PAR]; R9) --------- */
float oracle_fp16_decode(uint16_t code)
{
    uint32_t e = (code >> 10) & 0x1Fu, f = code & 0x3FFu;
    float mag;
    if (e == 31u)
        mag = (f == 0u) ? INFINITY : NAN;
    else
        mag = fp16_mag[code & 0x7FFFu];
    return (code & 0x8000u) ? -mag : mag;
}

uint16_t oracle_fp16_encode(float x)
{
    if (isnan(x))
        return 0;
    uint32_t mag = nearest_code(fp16_mag, 31u << 10, fabsf(x));
    return (uint16_t)((signbit(x) ? 0x8000u : 0u) | mag);
}

/* ---- bfloat16 output of the blockwise mode ([KB], p_out.to(bfloat16)) ---
 * IEEE round to nearest even.  A bfloat16 value is a binary32 value whose low
 * 16 bits are zero, so the magnitude code c stands for the float with bits
 * c << 16; the code 0x7F80 stands for 2^128 in the comparison (overflow to
 * Inf happens exactly as unbounded-exponent rounding says).  NaN -> 0x7FC0. */
static double bf16_code_value(uint32_t c)
{
    if (c >= 0x7F80u)
        return ldexp(1.0, 128);
    uint32_t bits = c << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

uint16_t oracle_bf16_round(float x)
{
    if (isnan(x))
        return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    float ax = fabsf(x);
    if (isinf(ax))
        return sign | 0x7F80u;
    uint32_t bits;
    memcpy(&bits, &ax, sizeof bits);
    uint32_t lo = bits >> 16; /* largest bfloat16 magnitude <= ax */
    double below = (double)ax - bf16_code_value(lo);
    if (below == 0.0)
        return sign | (uint16_t)lo;
    double above = bf16_code_value(lo + 1u) - (double)ax;
    uint32_t pick;
    if (below < above)
        pick = lo;
    else if (above < below)
        pick = lo + 1u;
    else
        pick = (lo % 2u == 0u) ? lo : lo + 1u;
    return sign | (uint16_t)pick;
}

/* ---------------------------------------------------------------------------
 * Hyperparameter scalars (R10).  [KB] forms 1-beta, beta^step, lr/bc1 and
 * 1-lr*wd in double precision and meets the FP32 tensors with them; here each
 * is formed in double and rounded once to FP32.
 * ------------------------------------------------------------------------- */
typedef struct {
    float b1;  /* beta1                          */
    float b2;  /* beta2                          */
    float c1;  /* 1 - beta1                      */
    float c2;  /* 1 - beta2                      */
    float bc2; /* 1 - beta2^step                 */
    float ss;  /* lr / (1 - beta1^step)          */
    float dk;  /* 1 - lr * wd  (decoupled decay) */
    float ef;  /* eps                            */
} oracle_hyper;

static oracle_hyper make_hyper(int64_t step, double lr, double beta1, double beta2,
                               double eps, double wd)
{
    oracle_hyper h;
    h.b1 = (float)beta1;
    h.b2 = (float)beta2;
    h.c1 = (float)(1.0 - beta1);
    h.c2 = (float)(1.0 - beta2);
    h.bc2 = (float)(1.0 - pow(beta2, (double)step));
    h.ss = (float)(lr / (1.0 - pow(beta1, (double)step)));
    h.dk = (float)(1.0 - lr * wd);
    h.ef = (float)eps;
    return h;
}

void oracle_hyperparams(int64_t step, double lr, double beta1, double beta2, double eps,
                        double wd, float out[8])
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    out[0] = h.b1; out[1] = h.b2; out[2] = h.c1; out[3] = h.c2;
    out[4] = h.bc2; out[5] = h.ss; out[6] = h.dk; out[7] = h.ef;
}

/* One AdamW element in FP32 ([TA] recurrences; [KB] operation order):
 *   m' = beta1*m + (1-beta1)*g
 *   v' = beta2*v + ((1-beta2)*g)*g
 *   p' = p*(1-lr*wd) - ((lr/bc1)*m') / (sqrt(v'/bc2) + eps)
 * Each line is one binary32 operation. */
static void adamw_element(float p, float g, float m, float v, const oracle_hyper *h,
                          float *p_new, float *m_new, float *v_new)
{
    float m1 = h->b1 * m;
    float m2 = h->c1 * g;
    float mn = m1 + m2;
    float t = h->c2 * g;
    float t2 = t * g;
    float v1 = h->b2 * v;
    float vn = v1 + t2;
    float q = vn / h->bc2;
    float s = sqrtf(q);
    float den = s + h->ef;
    float u = h->ss * mn;
    float upd = u / den;
    float pd = p * h->dk;
    *p_new = pd - upd;
    *m_new = mn;
    *v_new = vn;
}

static int nonfinite3(float a, float b, float c)
{
    return !isfinite(a) || !isfinite(b) || !isfinite(c);
}

/* Single AdamW element for tests (FP32 in, FP32 out). */
void oracle_adamw_element(float p, float g, float m, float v, int64_t step, double lr,
                          double beta1, double beta2, double eps, double wd, float out[3])
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    adamw_element(p, g, m, v, &h, &out[0], &out[1], &out[2]);
}

/* ---- Packed E4 step ([PAR], [PAC]) --------------------------------------
 * Decode m (low lane) and the uncorrected RMS r (high lane), v = r*r, FP32
 * update, then encode m' and sqrt(v') into the next word.  p and state are
 * updated in place.  Returns the number of elements whose p', m' or v' is not
 * finite. */
uint64_t oracle_step_packed_e4(float *p, const float *g, uint32_t *state, int64_t n,
                               int64_t step, double lr, double beta1, double beta2,
                               double eps, double wd)
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    uint64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t w = state[i];
        float m = oracle_e4m11_decode((uint16_t)(w & 0xFFFFu));
        float r = oracle_e4m12_decode((uint16_t)(w >> 16));
        float v = r * r;
        float pn, mn, vn;
        adamw_element(p[i], g[i], m, v, &h, &pn, &mn, &vn);
        float rn = sqrtf(vn);
        state[i] = ((uint32_t)oracle_e4m12_encode(rn) << 16) | oracle_e4m11_encode(mn);
        p[i] = pn;
        bad += (uint64_t)nonfinite3(pn, mn, vn);
    }
    return bad;
}

/* ---- Packed FP16-first / FP16-RMS comparison mode ([PAR]; R9) ---------- */
uint64_t oracle_step_packed_fp16(float *p, const float *g, uint32_t *state, int64_t n,
                                 int64_t step, double lr, double beta1, double beta2,
                                 double eps, double wd)
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    uint64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t w = state[i];
        float m = oracle_fp16_decode((uint16_t)(w & 0xFFFFu));
        float r = oracle_fp16_decode((uint16_t)(w >> 16));
        float v = r * r;
        float pn, mn, vn;
        adamw_element(p[i], g[i], m, v, &h, &pn, &mn, &vn);
        float rn = sqrtf(vn);
        state[i] = ((uint32_t)oracle_fp16_encode(rn) << 16) | oracle_fp16_encode(mn);
        p[i] = pn;
        bad += (uint64_t)nonfinite3(pn, mn, vn);
    }
    return bad;
}

/* ---- Ordinary FP32 AdamW comparison mode ([PAR]; [TA]; [KB]) ----------- */
uint64_t oracle_step_fp32(float *p, const float *g, float *m, float *v, int64_t n,
                          int64_t step, double lr, double beta1, double beta2, double eps,
                          double wd)
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    uint64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        float pn, mn, vn;
        adamw_element(p[i], g[i], m[i], v[i], &h, &pn, &mn, &vn);
        p[i] = pn;
        m[i] = mn;
        v[i] = vn;
        bad += (uint64_t)nonfinite3(pn, mn, vn);
    }
    return bad;
}

/* ---- Standalone packed-state codecs (E4 and FP16 words) ----------------- */
uint64_t oracle_encode_state_e4(const float *m, const float *rms, uint32_t *word, int64_t n)
{
    uint64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        word[i] = ((uint32_t)oracle_e4m12_encode(rms[i]) << 16) | oracle_e4m11_encode(m[i]);
        bad += (uint64_t)(!isfinite(m[i]) || !isfinite(rms[i]));
    }
    return bad;
}

void oracle_decode_state_e4(const uint32_t *word, float *m, float *rms, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        m[i] = oracle_e4m11_decode((uint16_t)(word[i] & 0xFFFFu));
        rms[i] = oracle_e4m12_decode((uint16_t)(word[i] >> 16));
    }
}

uint64_t oracle_encode_state_fp16(const float *m, const float *rms, uint32_t *word, int64_t n)
{
    uint64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        word[i] = ((uint32_t)oracle_fp16_encode(rms[i]) << 16) | oracle_fp16_encode(m[i]);
        bad += (uint64_t)(!isfinite(m[i]) || !isfinite(rms[i]));
    }
    return bad;
}

void oracle_decode_state_fp16(const uint32_t *word, float *m, float *rms, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        m[i] = oracle_fp16_decode((uint16_t)(word[i] & 0xFFFFu));
        rms[i] = oracle_fp16_decode((uint16_t)(word[i] >> 16));
    }
}

/* Array forms of the lane codecs, for the exhaustive format tests. */
void oracle_e4m11_encode_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m11_encode(x[i]);
}
void oracle_e4m12_encode_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m12_encode(x[i]);
}
void oracle_fp16_encode_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_encode(x[i]);
}
void oracle_e4m11_decode_array(const uint16_t *c, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m11_decode(c[i]);
}
void oracle_e4m12_decode_array(const uint16_t *c, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m12_decode(c[i]);
}
void oracle_fp16_decode_array(const uint16_t *c, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_decode(c[i]);
}
void oracle_bf16_round_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

/* ---------------------------------------------------------------------------
 * 8-bit blockwise mode ([KB]).
 * ------------------------------------------------------------------------- */
#define BLOCK 2048
#define ABSMAX_FLOOR 1e-30f

/* _requantise for one block of cnt <= BLOCK values: absmax = max |x| (NaN
 * propagates, R11); c = x / max(absmax, 1e-30); code = number of midpoints
 * strictly below c, which is the nearest map entry with an exact midpoint tie
 * going to the lower entry.  The stored absmax is the unclamped maximum. */
static void requantise_block(const float *x, int64_t cnt, const float *mid, uint8_t *code,
                             float *absmax_out)
{
    float a = 0.0f;
    for (int64_t i = 0; i < cnt; ++i) {
        float ax = fabsf(x[i]);
        if (isnan(a))
            break;
        if (isnan(ax) || ax > a)
            a = ax;
    }
    float scale = isnan(a) ? a : (a > ABSMAX_FLOOR ? a : ABSMAX_FLOOR);
    for (int64_t i = 0; i < cnt; ++i) {
        float c = x[i] / scale;
        int k = 0;
        for (int j = 0; j < 255; ++j)
            if (mid[j] < c)
                ++k;
        code[i] = (uint8_t)k;
    }
    *absmax_out = a;
}

/* The 255 midpoints of an ascending 256-entry map, each (q[i] + q[i+1]) * 0.5
 * in binary32. */
static void map_midpoints(const float *qmap, float *mid)
{
    for (int j = 0; j < 255; ++j) {
        float s = qmap[j] + qmap[j + 1];
        mid[j] = s * 0.5f;
    }
}

/* Requantise n values in blocks of 2048 (the last block may be short). */
void oracle_requantise(const float *x, int64_t n, const float *qmap, uint8_t *code,
                       float *absmax)
{
    float mid[255];
    map_midpoints(qmap, mid);
    for (int64_t b = 0; b * BLOCK < n; ++b) {
        int64_t lo = b * BLOCK;
        int64_t cnt = (n - lo < BLOCK) ? n - lo : BLOCK;
        requantise_block(x + lo, cnt, mid, code + lo, &absmax[b]);
    }
}

/* quantized_adamw_step: dequantise both moments through their maps and block
 * absmax, FP32 AdamW update, BF16 parameter output, then requantise the new
 * moments with fresh block absmax values.  p and g are read only; codes and
 * absmax arrays are replaced in place. */
uint64_t oracle_step_blockwise8(const float *p, const float *g, uint16_t *p_bf16,
                                uint8_t *m_code, float *m_absmax, uint8_t *v_code,
                                float *v_absmax, const float *qmap1, const float *qmap2,
                                int64_t n, int64_t step, double lr, double beta1,
                                double beta2, double eps, double wd)
{
    oracle_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    float mid1[255], mid2[255];
    map_midpoints(qmap1, mid1);
    map_midpoints(qmap2, mid2);
    static _Thread_local float mblk[BLOCK], vblk[BLOCK];
    uint64_t bad = 0;
    for (int64_t b = 0; b * BLOCK < n; ++b) {
        int64_t lo = b * BLOCK;
        int64_t cnt = (n - lo < BLOCK) ? n - lo : BLOCK;
        float am = m_absmax[b], av = v_absmax[b];
        for (int64_t k = 0; k < cnt; ++k) {
            int64_t i = lo + k;
            float m = qmap1[m_code[i]] * am;
            float v = qmap2[v_code[i]] * av;
            float pn, mn, vn;
            adamw_element(p[i], g[i], m, v, &h, &pn, &mn, &vn);
            p_bf16[i] = oracle_bf16_round(pn);
            mblk[k] = mn;
            vblk[k] = vn;
            bad += (uint64_t)nonfinite3(pn, mn, vn);
        }
        requantise_block(mblk, cnt, mid1, m_code + lo, &m_absmax[b]);
        requantise_block(vblk, cnt, mid2, v_code + lo, &v_absmax[b]);
    }
    return bad;
}
