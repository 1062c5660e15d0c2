/*
 * turbo.c -- plain, slow, scalar CPU oracle for the TurboAdam-style update:
 * the first moment persisted with UState, the second with 1Q.
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c (built into the same library): the
 * tests, the smoke check and bench.py's CPU-baseline leg are the only code
 * that may load it; the product path never calls it and shares no source.
 *
 * What it follows: the "TurboAdam" README (turboadam 0.2.0), "How it works":
 *   [UST] "UState: first-moment compression": the first moment is stored in
 *         normalised Adam update units q_t = (m_t / (1 - beta1^t)) /
 *         (sqrt(v_persisted_t / (1 - beta2^t)) + eps); a four-level packed
 *         code (2 bits per value), one bf16 mean per 64 values, and per tensor
 *         a decode scale, an encode scale and an RMS accumulator (12 bytes);
 *         each decoded mean block is recentred so that its stored bf16 mean is
 *         preserved; antithetic stochastic rounding; a one-step-lagged tensor
 *         scale with factor 1.1; beta1^2 < beta2 is required.
 *   [1Q]  "1Q: second-moment compression": per block of 128 values, packed
 *         4-bit indices on a logarithmic grid between two fp16 log endpoints;
 *         stochastic rounding between decoded positive values, from a counter
 *         hash (no stored random state).
 *   [UPD] "The AdamW update remains AdamW": m, v, the decoupled-decay update
 *         with bias corrections, from fp32 transient moments.
 *   [FUS] "Fused CUDA path": decode both states, rebuild the prior first
 *         moment in the persisted second-moment frame, form the fp32 moments,
 *         update the parameter, recompress the second moment with 1Q, then
 *         encode the next UState payload; a finaliser rotates the UState scale
 *         and clears the RMS accumulator.
 *   Memory table of the same README: 131,072 values hold 36,876 bytes of UState
 *   (2 bits per value + one bf16 per 64 + 12 bytes) and 69,632 bytes of 1Q (4
 *   bits per value + two fp16 per 128): the layouts below.
 *
 * Readings taken where the page is silent (all listed in the design notes):
 *   T1  1Q grid.  Index 0 decodes to 0; indices 1..K (K = 2^bits - 1) are the
 *       logarithmic grid from 2^lo to 2^hi, uniform in the binary32 bit
 *       pattern (a piecewise-linear log2, exact at powers of two):
 *       bits(level k) = B(lo) + floor(((B(hi) - B(lo)) * (k - 1) + (K-1)/2)
 *       / (K - 1)), B(e) = the bits of 2^e (e >= -149).  lo and hi are the
 *       integer binary exponents that bracket the block's positive values
 *       (2^lo <= smallest, largest <= 2^hi), held exactly as the fp16 log
 *       endpoints; a block with no positive value stores lo = hi = 0 and all
 *       indices 0.
 *   T2  1Q rounding.  v = 0 -> index 0; v on a level -> that level; else the
 *       bracketing levels d_j < v < d_(j+1) and index j+1 when u < (v - d_j)
 *       / (d_(j+1) - d_j), else j (unbiased in value); v above the top level
 *       (+Inf, or beyond 2^127) -> K.  A NaN or negative v -> index 0 (a NaN
 *       element counts as non-finite through v).  The stored width is 4 bits
 *       (the page's default; K = 15), two indices per byte.
 *   T3  Counter hash.  SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast
 *       splittable pseudorandom number generators", OOPSLA 2014; the public
 *       splitmix64 generator): output number c+1 of the generator seeded with
 *       `seed`, at counter c = step << 42 | stream << 40 | (index >> 1), is
 *       mix64(seed + (c + 1) * 0x9E3779B97F4A7C15); each output serves two
 *       indices: u = (bits 40..63 of it) * 2^-24 for an even index, (bits
 *       16..39) * 2^-24 for the odd one after it, in [0, 1).  Stream 1
 *       rounds 1Q, stream 2 UState.
 *   T4  UState code.  Four levels L = {-1.5, -0.5, 0.5, 1.5} in units of the
 *       encode scale s: y = r / s (0 when s = 0), z = clamp(y + 1.5, 0, 3),
 *       j = min(floor(z), 2), code = j + 1 when u < z - j, else j.  Antithetic:
 *       elements 2k and 2k+1 share u from counter index k, the odd one using
 *       1 - u.
 *   T5  UState decode.  d_i = s_dec * L[c_i]; per 64-value mean block of c
 *       values, delta = (s_dec * S) / (2c) with S the integer sum of 2*L[c_i];
 *       q_i = mu + (d_i - delta), mu the stored bf16 mean: the decoded block's
 *       mean is mu up to the rounding of the three operations.
 *   T6  UState mean.  The mean of q over a mean block is its sum taken as a
 *       pairwise tree over the 64 positions (adjacent pairs first, missing
 *       positions of a short last block as 0) divided by the number of
 *       values, rounded to bf16 (nearest even).  The residual is r = q - mu.
 *   T7  Scales.  The RMS accumulator adds r^2 over the tensor (float, in
 *       element order here; a parallel sum differs by rounding).  The
 *       finaliser sets s_dec <- s_enc, s_enc <- factor * sqrt(acc / n),
 *       acc <- 0.  All three start at 0, as do every code, mean, index and
 *       endpoint: the initial state decodes to m = v = 0.
 *   T8  Prior first moment.  m_(t-1) = (q * (sqrt(v_dec / bc2_(t-1)) + eps))
 *       * bc1_(t-1) with v_dec the decoded 1Q value (0 at step 1).  The new
 *       moments and the update are the FP32 element of oracle.c in its order;
 *       q_t uses the 1Q value the next step will decode.
 *   T9  Blocks start at the tensor's element 0; the last storage and mean
 *       blocks may be short.
 *
 * Build: compiled with oracle.c (gcc -std=c11 -O2 -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TURBO_BLOCK 128 /* 1Q storage block */
#define TURBO_MEAN 64   /* UState mean block */

/* ---- counter hash (T3) ---------------------------------------------------- */
uint64_t oracle_splitmix64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t oracle_splitmix64_at(uint64_t seed, uint64_t counter)
{
    return oracle_splitmix64_mix(seed + (counter + 1u) * 0x9E3779B97F4A7C15ull);
}

float oracle_turbo_uniform(uint64_t seed, int64_t step, uint32_t stream, uint64_t index)
{
    uint64_t c = ((uint64_t)step << 42) | ((uint64_t)stream << 40) | (index >> 1);
    uint64_t h = oracle_splitmix64_at(seed, c);
    uint64_t field = (index & 1u) ? (h >> 16) & 0xFFFFFFu : h >> 40;
    return (float)field * 0x1p-24f;
}

/* ---- 1Q (T1, T2) ------------------------------------------------------------ */
static float float_of(uint32_t u)
{
    float x;
    memcpy(&x, &u, 4);
    return x;
}

/* bits of 2^e, e in [-149, 127] */
static uint32_t pow2_bits(int e)
{
    if (e >= -126)
        return (uint32_t)(e + 127) << 23;
    return 1u << (e + 149);
}

/* Level k (1..K) of the grid [2^lo, 2^hi]; level 0 is 0. */
float oracle_q1_level(int lo, int hi, int bits, int k)
{
    if (k == 0)
        return 0.0f;
    int K = (1 << bits) - 1;
    uint64_t blo = pow2_bits(lo), bhi = pow2_bits(hi);
    uint64_t num = (bhi - blo) * (uint64_t)(k - 1) + (uint64_t)((K - 1) / 2);
    return float_of((uint32_t)(blo + num / (uint64_t)(K - 1)));
}

/* binary exponent e of positive finite x: 2^e <= x < 2^(e+1) */
static int exponent_of(float x)
{
    int e;
    frexpf(x, &e); /* x = f * 2^e, f in [0.5, 1) */
    return e - 1;
}

/* Endpoints of a block (T1): lo, hi bracket the positive values; 0, 0 if none. */
void oracle_q1_endpoints(const float *v, int64_t count, int *lo, int *hi)
{
    float mn = 0.0f, mx = 0.0f;
    int any = 0;
    for (int64_t i = 0; i < count; ++i) {
        float x = v[i];
        if (x > 0.0f && x <= 3.4028234663852886e38f) {
            if (!any || x < mn)
                mn = x;
            if (!any || x > mx)
                mx = x;
            any = 1;
        }
    }
    if (!any) {
        *lo = 0;
        *hi = 0;
        return;
    }
    *lo = exponent_of(mn);
    int e = exponent_of(mx);
    *hi = (mx == ldexpf(1.0f, e)) ? e : e + 1;
    if (*hi > 127) /* largest finite values: 2^128 is not a float; clamp */
        *hi = 127;
}

/* Index of v on the grid (T2) with uniform u. */
int oracle_q1_index(float v, int lo, int hi, int bits, float u)
{
    if (!(v > 0.0f))
        return 0;
    int K = (1 << bits) - 1;
    int j = 1;
    while (j < K && oracle_q1_level(lo, hi, bits, j + 1) <= v)
        ++j;
    float dj = oracle_q1_level(lo, hi, bits, j);
    if (v == dj || j == K)
        return j;
    float dn = oracle_q1_level(lo, hi, bits, j + 1);
    float p = (v - dj) / (dn - dj);
    return (u < p) ? j + 1 : j;
}

/* fp16 bits of an integer exponent in [-149, 127] (exact) and back */
static uint16_t fp16_of_int(int e)
{
    if (e == 0)
        return 0;
    uint16_t s = e < 0 ? 0x8000u : 0u;
    int a = e < 0 ? -e : e;
    int k = 0;
    while ((a >> (k + 1)) != 0)
        ++k; /* 2^k <= a < 2^(k+1), k <= 7 */
    uint16_t frac = (uint16_t)(((a - (1 << k)) << (10 - k)) & 0x3FF);
    return (uint16_t)(s | (uint16_t)((k + 15) << 10) | frac);
}

static int int_of_fp16(uint16_t h)
{
    if ((h & 0x7FFFu) == 0)
        return 0;
    int k = ((h >> 10) & 0x1F) - 15;
    int a = (1 << k) + ((h & 0x3FF) >> (10 - k));
    return (h & 0x8000u) ? -a : a;
}

uint16_t oracle_q1_endpoint_code(int e) { return fp16_of_int(e); }
int oracle_q1_endpoint_value(uint16_t h) { return int_of_fp16(h); }

/* bfloat16 rounding: oracle.c's (pinned against torch) */
uint16_t oracle_bf16_round(float x);

static float bf16_value(uint16_t h) { return float_of((uint32_t)h << 16); }

/* ---- UState (T4-T6) --------------------------------------------------------- */
static const float ULEVEL[4] = {-1.5f, -0.5f, 0.5f, 1.5f};
static const int ULEVEL2[4] = {-3, -1, 1, 3};

int oracle_ustate_code(float r, float s, float u)
{
    float y = (s > 0.0f) ? r / s : 0.0f;
    float z = y + 1.5f;
    if (!(z > 0.0f))
        z = 0.0f; /* also NaN -> 0 */
    if (z > 3.0f)
        z = 3.0f;
    int j = (int)floorf(z);
    if (j > 2)
        j = 2;
    float frac = z - (float)j;
    return (u < frac) ? j + 1 : j;
}

/* pairwise tree sum over 64 positions, adjacent pairs first (T6) */
static float tree_sum64(const float *x)
{
    float t[TURBO_MEAN];
    for (int i = 0; i < TURBO_MEAN; ++i)
        t[i] = x[i];
    for (int w = TURBO_MEAN; w > 1; w /= 2)
        for (int i = 0; i < w / 2; ++i)
            t[i] = t[2 * i] + t[2 * i + 1];
    return t[0];
}

/* ---- decoding the prior moments ([FUS] steps 1 and 2; T5, T8) ---------------- */
/* m_prev[j], v_dec[j] of elements i0 .. i0+cnt-1 (one 128-block). */
static void decode_block(int64_t i0, int64_t cnt, const uint8_t *ucode, const uint16_t *umean,
                         float sdec, const uint8_t *vidx, const uint16_t *vend, int64_t step,
                         double beta1, double beta2, float ef, float *m_prev, float *v_dec)
{
    const int bits = 4;
    float bc1p = (float)(1.0 - pow(beta1, (double)(step - 1)));
    float bc2p = (float)(1.0 - pow(beta2, (double)(step - 1)));
    int64_t b = i0 / TURBO_BLOCK;
    int lo = int_of_fp16(vend[2 * b]), hi = int_of_fp16(vend[2 * b + 1]);
    for (int64_t k = 0; k < cnt; k += TURBO_MEAN) {
        int64_t c = cnt - k < TURBO_MEAN ? cnt - k : TURBO_MEAN;
        int S = 0;
        for (int64_t j = 0; j < c; ++j) {
            int64_t i = i0 + k + j;
            S += ULEVEL2[(ucode[i / 4] >> (2 * (i % 4))) & 3u];
        }
        float delta = (sdec * (float)S) / (float)(2 * c);
        float mu = bf16_value(umean[(i0 + k) / TURBO_MEAN]);
        for (int64_t j = 0; j < c; ++j) {
            int64_t i = i0 + k + j;
            int code = (ucode[i / 4] >> (2 * (i % 4))) & 3u;
            int vi = (vidx[i / 2] >> (4 * (i % 2))) & 15u;
            float v = oracle_q1_level(lo, hi, bits, vi);
            float d = sdec * ULEVEL[code];
            float q = mu + (d - delta);
            float m = 0.0f;
            if (step > 1) {
                float den = sqrtf(v / bc2p) + ef;
                m = (q * den) * bc1p;
            }
            m_prev[k + j] = m;
            v_dec[k + j] = v;
        }
    }
}

/* The prior moments the step at `step` would decode from a state (tests). */
void oracle_turbo_decode(int64_t n, const uint8_t *ucode, const uint16_t *umean,
                         const float *uscal, const uint8_t *vidx, const uint16_t *vend,
                         int64_t step, double beta1, double beta2, double eps, float *m_prev,
                         float *v_dec)
{
    for (int64_t i0 = 0; i0 < n; i0 += TURBO_BLOCK) {
        int64_t cnt = n - i0 < TURBO_BLOCK ? n - i0 : TURBO_BLOCK;
        decode_block(i0, cnt, ucode, umean, uscal[0], vidx, vend, step, beta1, beta2,
                     (float)eps, m_prev + i0, v_dec + i0);
    }
}

/* ---- the step (T8, [FUS] order) ------------------------------------------ */
typedef struct {
    float b1, b2, c1, c2, bc2, ss, dk, ef;
} turbo_hyper;

static turbo_hyper make_hyper(int64_t step, double lr, double beta1, double beta2, double eps,
                              double wd)
{
    turbo_hyper h;
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

/*
 * One step over a tensor of n elements.  State layout:
 *   ucode  uint8[(n+3)/4]   2-bit UState codes, element i at bits 2*(i%4) of byte i/4
 *   umean  uint16[(n+63)/64] bf16 means
 *   uscal  float[3]          decode scale, encode scale, RMS accumulator (added to)
 *   vidx   uint8[(n+1)/2]    4-bit 1Q indices, element i in the low nibble of
 *                            byte i/2 when i is even, the high one when odd
 *   vend   uint16[2*nb]      fp16 endpoints (lo, hi) per 128-block
 * p is updated in place; returns the number of elements whose p', m or v is
 * not finite.  uscal[2] accumulates; call oracle_turbo_finalize after the step.
 */
/* The step over elements index0 .. index0+n-1 of a tensor (index0 a multiple
 * of the 128-value block; p, g and the state arrays start at element index0,
 * block index0 / 128 and mean block index0 / 64): the rounding counters take
 * the tensor's element indices.  Whole blocks are independent given the
 * scales, so a slice is updated as in the whole tensor, except the RMS
 * accumulator, which gathers the slice's squares only. */
uint64_t oracle_turbo_step_at(float *p, const float *g, int64_t n, uint8_t *ucode, uint16_t *umean,
                              float *uscal, uint8_t *vidx, uint16_t *vend, int64_t step,
                              double lr, double beta1, double beta2, double eps, double wd,
                              uint64_t seed, uint64_t index0);

uint64_t oracle_turbo_step(float *p, const float *g, int64_t n, uint8_t *ucode, uint16_t *umean,
                           float *uscal, uint8_t *vidx, uint16_t *vend, int64_t step,
                           double lr, double beta1, double beta2, double eps, double wd,
                           uint64_t seed)
{
    return oracle_turbo_step_at(p, g, n, ucode, umean, uscal, vidx, vend, step, lr, beta1, beta2,
                                eps, wd, seed, 0u);
}

uint64_t oracle_turbo_step_at(float *p, const float *g, int64_t n, uint8_t *ucode, uint16_t *umean,
                              float *uscal, uint8_t *vidx, uint16_t *vend, int64_t step,
                              double lr, double beta1, double beta2, double eps, double wd,
                              uint64_t seed, uint64_t index0)
{
    const int bits = 4;
    turbo_hyper h = make_hyper(step, lr, beta1, beta2, eps, wd);
    float bc1 = (float)(1.0 - pow(beta1, (double)step));
    float sdec = uscal[0], senc = uscal[1];
    float racc = uscal[2];
    uint64_t bad = 0;
    int64_t nb = (n + TURBO_BLOCK - 1) / TURBO_BLOCK;
    float mprev[TURBO_BLOCK], vdec[TURBO_BLOCK];
    float mnew[TURBO_BLOCK], vnew[TURBO_BLOCK], vhat[TURBO_BLOCK];
    for (int64_t b = 0; b < nb; ++b) {
        int64_t i0 = b * TURBO_BLOCK;
        int64_t cnt = n - i0 < TURBO_BLOCK ? n - i0 : TURBO_BLOCK;
        /* 1. decode both states; 2. rebuild the prior first moment */
        decode_block(i0, cnt, ucode, umean, sdec, vidx, vend, step, beta1, beta2, h.ef, mprev,
                     vdec);
        /* 3. the fp32 moments; 4. the update: the FP32 element of oracle.c, in its order */
        for (int64_t j = 0; j < cnt; ++j) {
            int64_t i = i0 + j;
            float m1 = h.b1 * mprev[j];
            float m2 = h.c1 * g[i];
            float mn = m1 + m2;
            float t = h.c2 * g[i];
            float t2 = t * g[i];
            float v1 = h.b2 * vdec[j];
            float vn = v1 + t2;
            float qq = vn / h.bc2;
            float s = sqrtf(qq);
            float den = s + h.ef;
            float u = h.ss * mn;
            float upd = u / den;
            float pd = p[i] * h.dk;
            p[i] = pd - upd;
            mnew[j] = mn;
            vnew[j] = vn;
            bad += (!isfinite(p[i]) || !isfinite(mn) || !isfinite(vn)) ? 1u : 0u;
        }
        /* 5. recompress v with 1Q */
        int nlo, nhi;
        oracle_q1_endpoints(vnew, cnt, &nlo, &nhi);
        vend[2 * b] = fp16_of_int(nlo);
        vend[2 * b + 1] = fp16_of_int(nhi);
        for (int64_t j = 0; j < cnt; ++j) {
            int64_t i = i0 + j;
            float u = oracle_turbo_uniform(seed, step, 1, index0 + (uint64_t)i);
            int vi = oracle_q1_index(vnew[j], nlo, nhi, bits, u);
            vidx[i / 2] = (uint8_t)((vidx[i / 2] & ~(15u << (4 * (i % 2)))) | ((unsigned)vi << (4 * (i % 2))));
            vhat[j] = oracle_q1_level(nlo, nhi, bits, vi);
        }
        /* 6. encode the next UState payload */
        for (int64_t k = 0; k < cnt; k += TURBO_MEAN) {
            int64_t c = cnt - k < TURBO_MEAN ? cnt - k : TURBO_MEAN;
            float qv[TURBO_MEAN];
            for (int64_t j = 0; j < TURBO_MEAN; ++j) {
                if (j < c) {
                    float den = sqrtf(vhat[k + j] / h.bc2) + h.ef;
                    qv[j] = (mnew[k + j] / bc1) / den;
                } else {
                    qv[j] = 0.0f;
                }
            }
            float mean = tree_sum64(qv) / (float)c;
            uint16_t mb = oracle_bf16_round(mean);
            umean[(i0 + k) / TURBO_MEAN] = mb;
            float mu = bf16_value(mb);
            for (int64_t j = 0; j < c; ++j) {
                int64_t i = i0 + k + j;
                float r = qv[j] - mu;
                float u = oracle_turbo_uniform(seed, step, 2, (index0 + (uint64_t)i) >> 1);
                if (i & 1)
                    u = 1.0f - u;
                int code = oracle_ustate_code(r, senc, u);
                ucode[i / 4] = (uint8_t)((ucode[i / 4] & ~(3u << (2 * (i % 4)))) | ((unsigned)code << (2 * (i % 4))));
                racc = racc + r * r;
            }
        }
    }
    uscal[2] = racc;
    return bad;
}

/* The finaliser (T7): rotate the scales, clear the accumulator. */
void oracle_turbo_finalize(float *uscal, int64_t n, double factor)
{
    float f = (float)factor;
    uscal[0] = uscal[1];
    uscal[1] = f * sqrtf(uscal[2] / (float)n);
    uscal[2] = 0.0f;
}

/* ---- array helpers for the tests ------------------------------------------ */
void oracle_turbo_uniform_array(uint64_t seed, int64_t step, uint32_t stream,
                                const uint64_t *index, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_turbo_uniform(seed, step, stream, index[i]);
}

void oracle_q1_levels(int lo, int hi, int bits, float *out)
{
    for (int k = 0; k < (1 << bits); ++k)
        out[k] = oracle_q1_level(lo, hi, bits, k);
}

void oracle_q1_index_array(const float *v, int64_t n, int lo, int hi, int bits, const float *u,
                           int32_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_q1_index(v[i], lo, hi, bits, u[i]);
}

void oracle_ustate_code_array(const float *r, int64_t n, float s, const float *u, int32_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_ustate_code(r[i], s, u[i]);
}

void oracle_q1_endpoints_pair(const float *v, int64_t count, int32_t *out)
{
    int lo, hi;
    oracle_q1_endpoints(v, count, &lo, &hi);
    out[0] = lo;
    out[1] = hi;
}
