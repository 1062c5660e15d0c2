// turbo.cuh -- the TurboAdam-style step: the first moment persisted with
// UState, the second with 1Q ("TurboAdam" README, turboadam 0.2.0, "How it
// works").  Included at the end of packedadam.cu (one translation unit: it
// uses that file's host helpers and the FP32 element of codecs.cuh).
//
// State of an n-element tensor (the README's memory table: 2 bits + one bf16
// per 64 values + 12 bytes of UState, 4 bits + two fp16 per 128 values of 1Q):
//   ucode  uint8[(n+3)/4]    2-bit UState codes, element i at bits 2*(i%4) of byte i/4
//   umean  uint16[(n+63)/64] bf16 mean of each 64-value mean block
//   uscal  float[3]          decode scale, encode scale, RMS accumulator
//   vidx   uint8[(n+1)/2]    4-bit 1Q indices, element i in nibble i%2 of byte i/2
//   vend   uint16[2*ceil(n/128)] fp16 log endpoints (lo, hi) of each 128-block
// Readings where the page is silent (listed in the header): the 1Q grid is
// uniform in the binary32 bit pattern between the integer binary exponents
// that bracket the block's positive values (exact, no transcendental
// function); index 0 is 0; stochastic rounding with u from SplitMix64 at a
// counter (step, stream, index / 2), each output's bits 40..63 serving the
// even index and bits 16..39 the odd one; UState levels {-1.5, -0.5, 0.5, 1.5} times
// the one-step-lagged encode scale, antithetic pairs (2k, 2k+1) share u and
// 1-u; block means are pairwise trees rounded to bf16; the finaliser rotates
// the scales (decode <- encode, encode <- factor * sqrt(acc / n), acc <- 0).
//
// Design.  One warp per 128-value storage block, lane l holding values
// 4l..4l+3 (16-byte loads of p and g; one code byte and one index half-word):
// the block's endpoints are warp min/max reductions over the binary32 bits of
// the positive values, the 15 levels of the old grid (decode) and of the new
// one live one per lane and are read by shuffles (the new one in a 4-step
// binary search), and a mean block's pairwise tree is the
// lane's own ((q0+q1)+(q2+q3)) followed by xor-shuffles over its 16 lanes --
// the same tree, since IEEE addition is commutative.  The RMS accumulator is
// one float atomic per warp (its sum order is the only thing that differs
// from a sequential evaluation).  Whole blocks take a body without bounds
// logic; a warp whose operands allow it takes the branch-free quotients and
// roots described above TurboFast.
#pragma once

namespace pa {

constexpr int kTurboBlock = 128;  // 1Q storage block
constexpr int kTurboMean = 64;    // UState mean block
constexpr int kTurboWarps = 8;    // warps (storage blocks in flight) per CTA
constexpr int kTurboThreads = kTurboWarps * 32;

struct TurboArgs {
    float *p;
    const float *g;
    int64_t n;
    uint8_t *ucode;
    uint16_t *umean;
    float *uscal;
    uint8_t *vidx;
    uint16_t *vend;
};

struct TurboScalars {
    Scalars s;        // the step's FP32 scalars (as every mode)
    float bc1;        // 1 - beta1^step
    float bc1p, bc2p; // 1 - beta1^(step-1), 1 - beta2^(step-1)
    uint64_t seed;
    int64_t step;
};

// ---- counter hash: SplitMix64 (Steele, Lea, Flood, OOPSLA 2014) at a counter
__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;  // SplitMix64's counter increment

// seed + (c + 1) * golden for the counter c of (step, stream, k), k the
// output's number in its stream (an index / 2): the input of the mix; k + j
// adds j * golden (k + j < 2^40 never carries into the stream and step fields)
__device__ __forceinline__ uint64_t turbo_counter(uint64_t seed, int64_t step, uint32_t stream,
                                                  uint64_t index)
{
    const uint64_t c = ((uint64_t)step << 42) | ((uint64_t)stream << 40) | index;
    return seed + (c + 1u) * kGolden;
}

// The two uniforms in [0, 1) on the 2^-24 grid that one output serves: bits
// 40..63 of the mix of z for the even index, bits 16..39 for the odd one.
__device__ __forceinline__ float2 turbo_uniform_pair(uint64_t z)
{
    const uint64_t h = splitmix64_mix(z);
    return make_float2(__uint2float_rn((uint32_t)(h >> 40)) * 0x1p-24f,
                       __uint2float_rn((uint32_t)(h >> 16) & 0xFFFFFFu) * 0x1p-24f);
}

// ---- 1Q grid ---------------------------------------------------------------------
__device__ __forceinline__ uint32_t pow2_bits(int e)
{
    return e >= -126 ? (uint32_t)(e + 127) << 23 : 1u << (e + 149);
}

// level k (0..15) of the grid [2^lo, 2^hi] given B(lo), B(hi): the bits
// B(lo) + floor((D (k-1) + 7) / 14), D = B(hi) - B(lo), in 32-bit arithmetic:
// with D = 14 Q + R the floor is Q (k-1) + floor((R (k-1) + 7) / 14), whose
// numerator is at most 13 * 14 + 7 = 189, where floor(t / 14) equals
// (t * 4682) >> 16 (checked for every t of that range).
__device__ __forceinline__ float q1_level(uint32_t blo, uint32_t bhi, int k)
{
    if (k <= 0)
        return 0.0f;
    const uint32_t d = bhi - blo, q = d / 14u, r = d - 14u * q, j = (uint32_t)(k - 1);
    return __uint_as_float(blo + q * j + (((r * j + 7u) * 4682u) >> 16));
}

// binary exponent of a positive finite float given its bits
__device__ __forceinline__ int exponent_of_bits(uint32_t b)
{
    return b >= 0x00800000u ? (int)(b >> 23) - 127 : (31 - __clz((int)b)) - 149;
}

__device__ __forceinline__ bool power_of_two_bits(uint32_t b)
{
    return b >= 0x00800000u ? (b & 0x007FFFFFu) == 0u : (b & (b - 1u)) == 0u;
}

// ---- UState code ------------------------------------------------------------------
// code of y = r / s (0 when s <= 0) with the uniform u
__device__ __forceinline__ uint32_t ustate_code_of(float y, float u)
{
    float z = __fadd_rn(y, 1.5f);
    z = z > 0.0f ? z : 0.0f;  // and NaN -> 0
    z = z > 3.0f ? 3.0f : z;
    int j = (int)floorf(z);
    j = j > 2 ? 2 : j;
    const float frac = __fsub_rn(z, (float)j);
    return (uint32_t)(j + (u < frac ? 1 : 0));
}

__device__ __forceinline__ int ulevel2(uint32_t c)  // 2 * {-1.5, -0.5, 0.5, 1.5}
{
    return 2 * (int)c - 3;
}

__device__ __forceinline__ float ulevel(uint32_t c)
{
    return (float)ulevel2(c) * 0.5f;
}

// Sum over the 16 lanes of this lane's half-warp, by xor-shuffles (a pairwise tree).
__device__ __forceinline__ float half_warp_tree(float x)
{
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, off));
    return x;
}

__device__ __forceinline__ int half_warp_sum(int x)
{
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
        x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    return x;
}

// ---- branch-free quotients ----------------------------------------------------------
// The denominators sqrt(level / bc2p) + eps (decode) and sqrt(level / bc2) +
// eps (encode) depend only on a grid level, so each lane forms the one of its
// level and elements fetch theirs by shuffle; a lane forms them branch-free
// too where the grid and bc2p (bc2) lie in the ranges below.  For the rest a
// warp replaces CUDA's correctly rounded divide and square root by
// the exact FMA forms of exact.cuh (Markstein's corrections, the residual
// root), same bits, where every operand lies in their ranges:
//  * launch (TurboFast::ok): bc2 in [2^-24, 1], bc1 in [2^-4, 1],
//    ss = lr/bc1 in [2^-20, 2^20], eps in [2^-40, 2^60];
//  * the block's v' (every v' finite, the positive ones in [2^-76, 2^99]) and so
//    the new grid [2^nlo, 2^nhi] with nlo >= -76, nhi <= 99: v'/bc2 below
//    2^123, its root in [2^-38, 2^62), den = root + eps in [2^-40, 2^63), the
//    encode's denominators in the same range; the 1Q fraction
//    (v - dj)/(dn - dj) has v - dj >= ulp(dj) >= 2^-99 and, the grid's levels
//    being at most 254/14 binades apart, a quotient above 2^-43;
//  * each lane's |m'|, which is 0 or NaN or in [2^-40, 2^40): u = ss*m' is 0 or
//    in [2^-60, 2^60] and u/den in [2^-123, 2^120]; t = m'/bc1 in [2^-40, 2^44)
//    and t/den in [2^-103, 2^84].  (A NaN operand gives NaN either way.)
//  * y = r/senc (TurboFast::sok, senc in [2^-20, 2^20]): |r| < 2^86 by the
//    bounds on t/den and on their bf16 mean, so nothing overflows; for
//    |r| >= 2^-100 the quotient is exact, and for smaller |r| both quotients
//    are below 2^-40 in magnitude, where RN(y + 1.5) = 1.5 for both and the
//    code is the same.
// Zero-signed quotients keep the dividend's sign (the divisors are positive).
struct TurboFast {
    float rb2, rb2p, rb1, rs;  // RN(1/bc2), RN(1/bc2p), RN(1/bc1), RN(1/senc)
    bool ok, sok, okp;         // okp: bc2p in [2^-24, 1] (the decode's levels)
};

__device__ __forceinline__ TurboFast turbo_fast_of(const TurboScalars &ts, float senc)
{
    const Scalars &s = ts.s;
    TurboFast f;
    const bool b2 = s.bc2 >= 0x1p-24f && s.bc2 <= 1.0f;
    const bool b1 = ts.bc1 >= 0x1p-4f && ts.bc1 <= 1.0f;
    f.ok = b2 && b1 && s.ss >= 0x1p-20f && s.ss <= 0x1p20f && s.ef >= 0x1p-40f && s.ef <= 0x1p60f;
    f.sok = senc >= 0x1p-20f && senc <= 0x1p20f;
    f.okp = ts.step > 1 && ts.bc2p >= 0x1p-24f && ts.bc2p <= 1.0f;
    f.rb2 = reciprocal_rn(b2 ? s.bc2 : 1.0f);
    f.rb2p = reciprocal_rn(f.okp ? ts.bc2p : 1.0f);
    f.rb1 = reciprocal_rn(b1 ? ts.bc1 : 1.0f);
    f.rs = reciprocal_rn(f.sok ? senc : 1.0f);
    return f;
}

// sqrt(x / b) (rb = RN(1/b)), IEEE or branch-free
template <bool BF>
__device__ __forceinline__ float root_of_quotient(float x, float b, float rb)
{
    if (BF)
        return sqrt_branch_free(quotient_by_reciprocal(x, b, rb));  // x = +0: +0
    return __fsqrt_rn(__fdiv_rn(x, b));
}

// c with the sign bits of a ORed in, lane by lane (a zero quotient keeps its
// dividend's sign; the divisors are positive)
__device__ __forceinline__ float2 with_sign_of(float2 c, float2 a)
{
    return make_float2(__uint_as_float(__float_as_uint(c.x) | (__float_as_uint(a.x) & 0x80000000u)),
                       __uint_as_float(__float_as_uint(c.y) | (__float_as_uint(a.y) & 0x80000000u)));
}

// What turbo_block carries from the moments to the recompression.
struct TurboLane {
    float p[4], mn[4], vn[4];
};

// The second half of a storage block (the update, 1Q and UState encode,
// stores), with the IEEE or the branch-free quotients.
template <bool WHOLE, bool BF>
__device__ __forceinline__ void turbo_encode(const TurboArgs &a, const TurboScalars &ts,
                                             const TurboFast &f, float senc, TurboLane &L,
                                             int64_t i0, int64_t e0, int valid, int mcount,
                                             int64_t mstart, uint32_t cbyte, uint32_t vhalf,
                                             uint32_t pmin, uint32_t pmax, const float u1[4],
                                             const float upair[2], uint32_t &bad, float &racc)
{
    const int lane = threadIdx.x & 31;
    const Scalars &s = ts.s;
    // ---- 4. the update (the FP32 element of every mode; pairs of elements
    //      in packed arithmetic, each lane the scalar operations' bits)
    {
        const Pairs k = pairs_of(s);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const float2 vn = make_float2(L.vn[j], L.vn[j + 1]);
            const float2 nu = mul2(k.nss, make_float2(L.mn[j], L.mn[j + 1]));
            float2 nupd;
            if (BF) {
                nupd = pair_update_branch_free<false>(vn, nu, k, make_float2(-s.bc2, -s.bc2),
                                                      make_float2(f.rb2, f.rb2), nullptr);
            } else {
                nupd.x = __fdiv_rn(nu.x, __fadd_rn(root_of_quotient<false>(vn.x, s.bc2, f.rb2), s.ef));
                nupd.y = __fdiv_rn(nu.y, __fadd_rn(root_of_quotient<false>(vn.y, s.bc2, f.rb2), s.ef));
            }
#ifndef PA_FAST_MATH
            const float2 pn = add2x(mul2(make_float2(L.p[j], L.p[j + 1]), k.dk), nupd, k.one);
#else
            const float2 pn = fma2(make_float2(L.p[j], L.p[j + 1]), k.dk, nupd);  // as adamw_element
#endif
            L.p[j] = pn.x;
            L.p[j + 1] = pn.y;
        }
        if (!WHOLE) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < valid)
                    bad += any_nonfinite(Moments{L.p[j], L.mn[j], L.vn[j]});
        }
    }
    if (WHOLE) {  // the lane's four at once (packed FMAs; counted one by one only if any)
        const Moments2 o[2] = {{make_float2(L.p[0], L.p[1]), make_float2(L.mn[0], L.mn[1]), make_float2(L.vn[0], L.vn[1])},
                               {make_float2(L.p[2], L.p[3]), make_float2(L.mn[2], L.mn[3]), make_float2(L.vn[2], L.vn[3])}};
        bad += nonfinite_count4(o);
    }
    // ---- 5. recompress v with 1Q: endpoints from the block's positive values
    int nlo = 0, nhi = 0;
    if (pmax != 0u) {
        nlo = exponent_of_bits(pmin);
        const int e = exponent_of_bits(pmax);
        nhi = power_of_two_bits(pmax) ? e : e + 1;
        nhi = nhi > 127 ? 127 : nhi;
    }
    const uint32_t nblo = pow2_bits(nlo), nbhi = pow2_bits(nhi);
    // lane k holds level k of the new grid and the encode's denominator for it,
    // sqrt(level / bc2) + eps (the same value for every element that takes it);
    // on the branch-free arm also the reciprocals that the elements' quotients
    // take: RN(1/den) and, for k < 15, RN(1/(level k+1 - level k)) with that gap
    const int mylane = lane < 16 ? lane : 15;
    const float mylevel = q1_level(nblo, nbhi, mylane);
    const float myden = __fadd_rn(root_of_quotient<BF>(mylevel, s.bc2, f.rb2), s.ef);
    float myrden = 0.0f, mygap = 0.0f, myrgap = 0.0f;
    if (BF) {
        myrden = reciprocal_rn(myden);
        mygap = __fsub_rn(q1_level(nblo, nbhi, mylane < 15 ? mylane + 1 : 15), mylevel);
        myrgap = reciprocal_rn(mygap > 0.0f ? mygap : 1.0f);
    }
    // (the branch-free arm fetches negated levels, gaps and denominators: its
    // quotients take the divisor negated, exact.cuh's pair forms)
    const float mysel = BF ? -myden : myden;
    uint32_t nvhalf = 0;
    float den5[4], rden5[4];
    int kk[4];
    float ndj[4], ngap[4], rgap[4], frac[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // k = the number of levels 1..15 at most v: for positive v (>= level
        // 1) the largest such level; the probes stay within 1..15
        int k = 0;
#pragma unroll
        for (int step = 8; step >= 1; step >>= 1) {
            const int c = k + step;
            k = __shfl_sync(0xFFFFFFFFu, mylevel, c) <= L.vn[j] ? c : k;
        }
        kk[j] = k;
        if (BF) {
            ndj[j] = __shfl_sync(0xFFFFFFFFu, -mylevel, k);
            ngap[j] = __shfl_sync(0xFFFFFFFFu, -mygap, k);
            rgap[j] = __shfl_sync(0xFFFFFFFFu, myrgap, k);
        }
    }
    if (BF) {  // the fractions (v - level k) / gap k of all four, in pairs
        const float2 one = one_pair();
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const float2 d = add2x(make_float2(L.vn[j], L.vn[j + 1]), make_float2(ndj[j], ndj[j + 1]), one);
            const float2 fr = quotient_by_reciprocal2(d, make_float2(ngap[j], ngap[j + 1]),
                                                      make_float2(rgap[j], rgap[j + 1]));
            frac[j] = fr.x;
            frac[j + 1] = fr.y;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float v = L.vn[j];
        const int k = kk[j];
        int idx = 0;
        if (BF) {
            // (level 0 and a zero gap give fractions that are not used)
            if (v > 0.0f)
                idx = (v == -ndj[j] || k == 15) ? k : (u1[j] < frac[j] ? k + 1 : k);
        } else {
            const float dj = __shfl_sync(0xFFFFFFFFu, mylevel, k);
            const float dn = __shfl_sync(0xFFFFFFFFu, mylevel, k < 15 ? k + 1 : 15);
            if (v > 0.0f) {
                idx = k;
                if (!(v == dj || k == 15))
                    idx = u1[j] < __fdiv_rn(__fsub_rn(v, dj), __fsub_rn(dn, dj)) ? k + 1 : k;
            }
        }
        nvhalf |= (uint32_t)idx << (4 * j);
        den5[j] = __shfl_sync(0xFFFFFFFFu, mysel, idx);  // BF: -den
        if (BF)
            rden5[j] = __shfl_sync(0xFFFFFFFFu, myrden, idx);
    }
    // ---- 6. encode the next UState payload: q = (m'/bc1)/den
    float q[4];
    if (WHOLE && BF) {  // pairs of elements (each lane the scalar form's bits)
        const float2 nbc1 = make_float2(-ts.bc1, -ts.bc1), rb1 = make_float2(f.rb1, f.rb1);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const float2 mn = make_float2(L.mn[j], L.mn[j + 1]);
            const float2 t = with_sign_of(quotient_by_reciprocal2(mn, nbc1, rb1), mn);
            const float2 c = with_sign_of(quotient_by_reciprocal2(t, make_float2(den5[j], den5[j + 1]),
                                                                  make_float2(rden5[j], rden5[j + 1])),
                                          t);
            q[j] = c.x;
            q[j + 1] = c.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (WHOLE || j < valid) {
                const float t = BF ? __uint_as_float(__float_as_uint(quotient_by_reciprocal(L.mn[j], ts.bc1, f.rb1)) |
                                                     (__float_as_uint(L.mn[j]) & 0x80000000u))
                                   : __fdiv_rn(L.mn[j], ts.bc1);
                if (BF) {
                    const float c = quotient_by_reciprocal(t, -den5[j], rden5[j]);
                    q[j] = __uint_as_float(__float_as_uint(c) | (__float_as_uint(t) & 0x80000000u));
                } else {
                    q[j] = __fdiv_rn(t, den5[j]);
                }
            } else {
                q[j] = 0.0f;  // missing positions of a short block count as 0
            }
        }
    }
    const float tree = half_warp_tree(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])));
    // (dividing by 64 = multiplying by 2^-6: the same rounded result)
    const float mean = WHOLE ? __fmul_rn(tree, 0x1p-6f)
                             : (mcount > 0 ? __fdiv_rn(tree, (float)mcount) : 0.0f);
    const __nv_bfloat16 mb = __float2bfloat16_rn(mean);
    uint16_t mbits = *reinterpret_cast<const uint16_t *>(&mb);
    if (mean != mean)
        mbits = 0x7FC0u;
    const float mub = __uint_as_float((uint32_t)mbits << 16);
    uint32_t ncbyte = cbyte;
    float rsum = 0.0f;
    if (WHOLE && BF && f.sok) {  // (f.sok is uniform over the launch)
        // pairs: r = q - mean, y = r / senc, r*r; codes and the sum in order
        const float2 one = one_pair(), nmub = make_float2(-mub, -mub);
        const float2 nsenc = make_float2(-senc, -senc), rs = make_float2(f.rs, f.rs);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const float2 r = add2x(make_float2(q[j], q[j + 1]), nmub, one);
            const float2 y = quotient_by_reciprocal2(r, nsenc, rs);
            const float2 rr = mul2(r, r);
            const uint32_t c0 = ustate_code_of(y.x, upair[j >> 1]);
            const uint32_t c1 = ustate_code_of(y.y, __fsub_rn(1.0f, upair[j >> 1]));
            ncbyte = (ncbyte & ~(15u << (2 * j))) | (c0 << (2 * j)) | (c1 << (2 * j + 2));
            rsum = __fadd_rn(__fadd_rn(rsum, rr.x), rr.y);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (WHOLE || j < valid) {
                const float r = __fsub_rn(q[j], mub);
                const float u = (j & 1) ? __fsub_rn(1.0f, upair[j >> 1]) : upair[j >> 1];
                float y;
                if (BF && f.sok)  // uniform over the launch (|r| < 2^86 needs the BF bounds)
                    y = quotient_by_reciprocal(r, senc, f.rs);
                else
                    y = senc > 0.0f ? __fdiv_rn(r, senc) : 0.0f;
                const uint32_t c = ustate_code_of(y, u);
                ncbyte = (ncbyte & ~(3u << (2 * j))) | (c << (2 * j));
                rsum = __fadd_rn(rsum, __fmul_rn(r, r));
            }
        }
    }
    // ---- stores
    if (WHOLE || valid == 4) {
        *reinterpret_cast<float4 *>(a.p + e0) = make_float4(L.p[0], L.p[1], L.p[2], L.p[3]);
        a.ucode[e0 / 4] = (uint8_t)ncbyte;
        *reinterpret_cast<uint16_t *>(a.vidx + e0 / 2) = (uint16_t)nvhalf;
    } else if (valid > 0) {
        for (int j = 0; j < valid; ++j)
            a.p[e0 + j] = L.p[j];
        a.ucode[e0 / 4] = (uint8_t)ncbyte;
        // indices of elements past n keep their old nibbles
        const uint32_t keep = valid >= 4 ? 0u : (0xFFFFu << (4 * valid)) & 0xFFFFu;
        const uint32_t nv = (nvhalf & ~keep) | (vhalf & keep);
        a.vidx[e0 / 2] = (uint8_t)nv;
        if (valid > 2)
            a.vidx[e0 / 2 + 1] = (uint8_t)(nv >> 8);
    }
    if ((lane & 15) == 0 && (WHOLE || mcount > 0))
        a.umean[mstart / kTurboMean] = mbits;
    if (lane == 0) {
        const int64_t b = i0 / kTurboBlock;
        a.vend[2 * b] = __half_as_ushort(__int2half_rn(nlo));
        a.vend[2 * b + 1] = __half_as_ushort(__int2half_rn(nhi));
    }
    racc = __fadd_rn(racc, rsum);
}

// A lane's inputs for one storage block: its values, their codes and indices,
// the block's endpoints and its mean block's bf16 mean.
struct TurboIn {
    float p[4], g[4];
    uint32_t cbyte, vhalf;
    uint16_t vlo, vhi, mean;
};

template <bool WHOLE>
__device__ __forceinline__ TurboIn turbo_load(const TurboArgs &a, int64_t i0)
{
    const int lane = threadIdx.x & 31;
    const int64_t e0 = i0 + 4 * lane;
    const int valid = WHOLE ? 4 : (e0 >= a.n ? 0 : (a.n - e0 >= 4 ? 4 : (int)(a.n - e0)));
    TurboIn in;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        in.p[j] = in.g[j] = 0.0f;
    in.cbyte = in.vhalf = 0u;
    if (WHOLE || valid == 4) {
        const float4 pv = *reinterpret_cast<const float4 *>(a.p + e0);
        const float4 gv = __ldg(reinterpret_cast<const float4 *>(a.g + e0));
        in.p[0] = pv.x; in.p[1] = pv.y; in.p[2] = pv.z; in.p[3] = pv.w;
        in.g[0] = gv.x; in.g[1] = gv.y; in.g[2] = gv.z; in.g[3] = gv.w;
        in.cbyte = a.ucode[e0 / 4];
        in.vhalf = *reinterpret_cast<const uint16_t *>(a.vidx + e0 / 2);
    } else if (valid > 0) {
        for (int j = 0; j < valid; ++j) {
            in.p[j] = a.p[e0 + j];
            in.g[j] = a.g[e0 + j];
        }
        in.cbyte = a.ucode[e0 / 4];
        in.vhalf = a.vidx[e0 / 2] | (valid > 2 ? (uint32_t)a.vidx[e0 / 2 + 1] << 8 : 0u);
    }
    const int64_t b = i0 / kTurboBlock;
    in.vlo = a.vend[2 * b];
    in.vhi = a.vend[2 * b + 1];
    const int64_t mstart = i0 + kTurboMean * (lane >> 4);
    in.mean = (WHOLE || mstart < a.n) ? a.umean[mstart / kTurboMean] : (uint16_t)0;
    return in;
}

// One storage block (128 values from element i0) by one warp, from its loaded
// inputs.  WHOLE: all 128 values lie below n.
template <bool WHOLE>
__device__ __forceinline__ void turbo_block(const TurboArgs &a, const TurboScalars &ts,
                                            const TurboFast &f, float sdec, float senc, int64_t i0,
                                            const TurboIn &in, uint32_t &bad, float &racc)
{
    const int lane = threadIdx.x & 31;
    const int64_t e0 = i0 + 4 * lane;  // this lane's first element
    const int valid = WHOLE ? 4 : (e0 >= a.n ? 0 : (a.n - e0 >= 4 ? 4 : (int)(a.n - e0)));
    const Scalars &s = ts.s;
    // The rounding uniforms depend on the counters alone: formed here, where
    // they overlap the block's loads (2 % faster on GB300 than where they are
    // used; builds without the hashes ran 19 % faster).  Each hash output
    // serves two indices.  1Q: one uniform per value, two outputs for the
    // lane's four; UState: one per antithetic pair (2k, 2k+1), which share u
    // and 1-u, one output for the lane's two pairs (e0 is a multiple of 4).
    float u1[4], upair[2];
    {
        const uint64_t z1 = turbo_counter(ts.seed, ts.step, 1u, (uint64_t)e0 >> 1);
        const uint64_t z2 = turbo_counter(ts.seed, ts.step, 2u, (uint64_t)e0 >> 2);
        const float2 a = turbo_uniform_pair(z1), b = turbo_uniform_pair(z1 + kGolden);
        const float2 c = turbo_uniform_pair(z2);
        u1[0] = a.x;
        u1[1] = a.y;
        u1[2] = b.x;
        u1[3] = b.y;
        upair[0] = c.x;
        upair[1] = c.y;
    }
    TurboLane L;
    float g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        L.p[j] = in.p[j];
        g[j] = in.g[j];
    }
    const uint32_t cbyte = in.cbyte, vhalf = in.vhalf;
    const int lo = __half2int_rn(__ushort_as_half(in.vlo));
    const int hi = __half2int_rn(__ushort_as_half(in.vhi));
    const uint32_t blo = pow2_bits(lo), bhi = pow2_bits(hi);
    const int half = lane >> 4;  // mean block of this lane within the storage block
    const int64_t mstart = i0 + kTurboMean * half;
    const int mcount = WHOLE ? kTurboMean
                             : (mstart >= a.n ? 0 : (a.n - mstart >= kTurboMean ? kTurboMean : (int)(a.n - mstart)));
    // ---- 1. decode UState (recentred means) and 1Q (lane k holds old level k);
    //      2. the prior first moment
    int S = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (WHOLE || j < valid)
            S += ulevel2((cbyte >> (2 * j)) & 3u);
    S = half_warp_sum(S);
    const float mu = (WHOLE || mcount > 0) ? __uint_as_float((uint32_t)in.mean << 16) : 0.0f;
    const float delta = WHOLE ? __fmul_rn(__fmul_rn(sdec, (float)S), 0x1p-7f)  // / 128
                              : (mcount > 0 ? __fdiv_rn(__fmul_rn(sdec, (float)S), (float)(2 * mcount)) : 0.0f);
    // lane k holds level k of the old grid and the prior denominator for it,
    // sqrt(level / bc2p) + eps
    const float oldlevel = q1_level(blo, bhi, lane < 16 ? lane : 15);
    // (branch-free when the old grid lies in [2^-100, 2^99]: the level over
    // bc2p below 2^123, its root in the residual root's range)
    float oldden = 0.0f;
    if (ts.step > 1)
        oldden = __fadd_rn(f.okp && lo >= -100 && hi <= 99 ? root_of_quotient<true>(oldlevel, ts.bc2p, f.rb2p)
                                                            : root_of_quotient<false>(oldlevel, ts.bc2p, f.rb2p),
                           s.ef);
    // the recentred value mu + (sdec * level(c) - delta) of UState code c,
    // held by lane c of each half-warp (its mean block's) and fetched by shuffle
    const float qcode = __fadd_rn(mu, __fsub_rn(__fmul_rn(sdec, ulevel((uint32_t)lane & 3u)), delta));
    float mprev[4], vdec[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int idx = (int)((vhalf >> (4 * j)) & 15u);
        const float v = __shfl_sync(0xFFFFFFFFu, oldlevel, idx);
        const float den = __shfl_sync(0xFFFFFFFFu, oldden, idx);
        const float q = __shfl_sync(0xFFFFFFFFu, qcode, (lane & 16) | (int)((cbyte >> (2 * j)) & 3u));
        mprev[j] = ts.step > 1 ? __fmul_rn(__fmul_rn(q, den), ts.bc1p) : 0.0f;
        vdec[j] = v;
    }
    // ---- 3. the fp32 moments (pairs of elements in packed arithmetic, each
    //      lane the scalar b1*m + c1*g and b2*v + (c2*g)*g); the block's v'
    //      range; each lane's |m'| range
    {
        const float2 one = one_pair();
        const float2 b1 = make_float2(s.b1, s.b1), c1 = make_float2(s.c1, s.c1);
        const float2 b2 = make_float2(s.b2, s.b2), c2 = make_float2(s.c2, s.c2);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const float2 gp = make_float2(g[j], g[j + 1]);
            const float2 mn = add2x(mul2(b1, make_float2(mprev[j], mprev[j + 1])), mul2(c1, gp), one);
            const float2 vn = add2x(mul2(b2, make_float2(vdec[j], vdec[j + 1])), mul2(mul2(c2, gp), gp), one);
            L.mn[j] = mn.x;
            L.mn[j + 1] = mn.y;
            L.vn[j] = vn.x;
            L.vn[j + 1] = vn.y;
        }
    }
    uint32_t pmin = 0xFFFFFFFFu, pmax = 0u, vall = 0u;
    float mlo = INFINITY, mhi = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t bits = __float_as_uint(L.vn[j]);
        if (WHOLE || j < valid) {
            const bool pos = L.vn[j] > 0.0f && bits < 0x7F800000u;
            pmin = pos ? min(pmin, bits) : pmin;
            pmax = pos ? max(pmax, bits) : pmax;
            vall = max(vall, bits);
            mlo = fminf(mlo, fabsf(L.mn[j]));  // NaN ignored (NaN is NaN either way)
            mhi = fmaxf(mhi, fabsf(L.mn[j]));
        }
    }
    pmin = __reduce_min_sync(0xFFFFFFFFu, pmin);
    pmax = __reduce_max_sync(0xFFFFFFFFu, pmax);
    vall = __reduce_max_sync(0xFFFFFFFFu, vall);
    // positive v' in [2^-76, 2^99], none non-finite or negative; |m'| range
    const bool lane_ok = f.ok && (pmax == 0u || (pmin >= 0x19800000u && pmax <= 0x71000000u)) &&
                         vall <= 0x71000000u && mlo >= 0x1p-40f && mhi < 0x1p40f;
    if (__all_sync(0xFFFFFFFFu, lane_ok))
        turbo_encode<WHOLE, true>(a, ts, f, senc, L, i0, e0, valid, mcount, mstart, cbyte, vhalf,
                                  pmin, pmax, u1, upair, bad, racc);
    else
        turbo_encode<WHOLE, false>(a, ts, f, senc, L, i0, e0, valid, mcount, mstart, cbyte, vhalf,
                                   pmin, pmax, u1, upair, bad, racc);
}

// (three CTAs per SM with up to 80 registers: 2.3 % faster on GB300 than four
// CTAs at 64 registers once the update and the UState encode ran in packed
// pairs; before them four CTAs had been 4 % faster, and five lost again.)
__global__ void __launch_bounds__(kTurboThreads, 3)
turbo_step_kernel(const TurboArgs a, const TurboScalars ts, unsigned long long *nonfinite)
{
    const float sdec = a.uscal[0], senc = a.uscal[1];
    const int64_t nblocks = (a.n + kTurboBlock - 1) / kTurboBlock;
    const int64_t warp = (int64_t)blockIdx.x * kTurboWarps + (threadIdx.x >> 5);
    const int64_t warps = (int64_t)gridDim.x * kTurboWarps;
    const TurboFast f = turbo_fast_of(ts, senc);
    const int64_t nwhole = a.n / kTurboBlock;
    uint32_t bad = 0;
    float racc = 0.0f;
    // (Loading a warp's next block before computing the current one measured
    // 6 % slower on GB300.)
    int64_t b = warp;
    for (; b < nwhole; b += warps)  // uniform per warp
        turbo_block<true>(a, ts, f, sdec, senc, b * kTurboBlock, turbo_load<true>(a, b * kTurboBlock),
                          bad, racc);
    if (b < nblocks)  // the short last block
        turbo_block<false>(a, ts, f, sdec, senc, b * kTurboBlock, turbo_load<false>(a, b * kTurboBlock),
                           bad, racc);
    // the RMS accumulator: one atomic per warp
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        racc = __fadd_rn(racc, __shfl_xor_sync(0xFFFFFFFFu, racc, off));
    if ((threadIdx.x & 31) == 0 && racc != 0.0f)
        atomicAdd(a.uscal + 2, racc);
    flush_nonfinite(bad, nonfinite);
}

// The finaliser: decode scale <- encode scale, encode scale <- factor *
// sqrt(acc / n), acc <- 0.
__global__ void turbo_finalize_kernel(float *uscal, float nf, float factor)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const float acc = uscal[2];
        uscal[0] = uscal[1];
        uscal[1] = __fmul_rn(factor, __fsqrt_rn(__fdiv_rn(acc, nf)));
        uscal[2] = 0.0f;
    }
}

}  // namespace pa
