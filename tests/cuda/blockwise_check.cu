// GPU check of the blockwise requantiser's helpers (test code): the bucket
// search against the plain 8-step binary search for every binary32 c in
// [-1, 1], the FMA division by the block scale against __fdiv_rn on random
// (x, scale) pairs, the Newton-refined reciprocal (scalar and packed pair
// form) against __frcp_rn for every scale of the fast range, and whole codes (reciprocal, FMA quotient, bucket
// search, IEEE fix-up below the floor) against the count of midpoints below
// the IEEE quotient.  Kernels only add to counters and write the first
// mismatch into a fixed 4-word slot claimed with atomicCAS.
#include <cuda_runtime.h>
#include <cstdint>
#include "blockwise.cuh"

using namespace pa;

__device__ void note(unsigned long long *count, uint32_t *first, uint32_t a, uint32_t b, uint32_t got, uint32_t want)
{
    atomicAdd(count, 1ull);
    if (atomicCAS(first, 0u, 1u) == 0u) {
        first[1] = a; first[2] = b; first[3] = got ^ (want << 16);
    }
}

// every c in [-1, 1]: both signs, every binary32 pattern of magnitude <= 1
__global__ void search_all(const float *qmap, unsigned long long *count, uint32_t *first)
{
    __shared__ float q[256], mid[512];
    __shared__ uint8_t table[kBuckets];
    __shared__ uint32_t red[32];
    const int tid = threadIdx.x;
    q[tid] = qmap[tid];
    __syncthreads();
    mid[tid] = tid < 255 ? __fmul_rn(__fadd_rn(q[tid], q[tid + 1]), 0.5f) : INFINITY;
    mid[256 + tid] = INFINITY;
    __syncthreads();
    const int k = build_buckets(mid, table, red);
    __syncthreads();
    const uint64_t half = (uint64_t)0x3F800000u + 1;  // magnitudes 0 .. 1.0
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + tid; i < 2 * half; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t bits = i < half ? (uint32_t)i : 0x80000000u | (uint32_t)(i - half);
        const float c = __uint_as_float(bits);
        const uint32_t got = k <= 2 ? code_by_bucket<2>(mid, table, c, k) : code_by_bucket<0>(mid, table, c, k);
        const uint32_t want = (uint32_t)count_below(mid, c);
        if (got != want)
            note(count, first, __float_as_uint(c), 0, got, want);
    }
}

__device__ uint32_t mix32(uint64_t x)
{
    x ^= x >> 31; x *= 0x7fb5d329728ea185ull; x ^= x >> 27; x *= 0x81dadef4bc2dd44dull; x ^= x >> 33;
    return (uint32_t)x;
}

__global__ void divide_random(uint64_t n, uint64_t seed, unsigned long long *count, uint32_t *first)
{
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t r0 = mix32(3 * i + seed), r1 = mix32(3 * i + 1 + seed), r2 = mix32(3 * i + 2 + seed);
        // scale: a normal number in [2^-100, 2^100)
        const uint32_t sb = 0x0D800000u + r0 % 0x64000000u;
        // x: |x| <= scale, exponent up to 160 binades below, some zeros, random sign
        const uint32_t drop = (r1 >> 24) % 160u;
        uint32_t xb = (r1 & 0x007FFFFFu) | ((sb & 0x7F800000u) - (drop << 23) * ((sb >> 23) > drop));
        if ((sb >> 23) <= drop) xb = r1 & 0x007FFFFFu;  // subnormal x
        if (xb > sb) xb = sb;
        if ((r2 & 0xFFu) == 0u) xb = 0u;
        xb |= r2 & 0x80000000u;
        const float x = __uint_as_float(xb), s = __uint_as_float(sb);
        const float got = needs_ieee_divide(x, fast_quotient_floor(sb)) ? __fdiv_rn(x, s)
                                                                        : divide_by_scale_fma(x, s, __frcp_rn(s));
        const float want = __fdiv_rn(x, s);
        if (__float_as_uint(got) != __float_as_uint(want))
            note(count, first, xb, sb, __float_as_uint(got), __float_as_uint(want));
    }
}

extern "C" int run_search_all(const float *qmap_host, unsigned long long *count_host, uint32_t *first_host)
{
    float *q; unsigned long long *c; uint32_t *f;
    if (cudaMalloc(&q, 256 * 4) || cudaMalloc(&c, 8) || cudaMalloc(&f, 16)) return -1;
    cudaMemcpy(q, qmap_host, 256 * 4, cudaMemcpyHostToDevice);
    cudaMemset(c, 0, 8); cudaMemset(f, 0, 16);
    search_all<<<152 * 4, kThreadsPerBlockwiseCta>>>(q, c, f);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(count_host, c, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(first_host, f, 16, cudaMemcpyDeviceToHost);
    cudaFree(q); cudaFree(c); cudaFree(f);
    return e;
}

// every scale bit pattern of [2^-100, 2^100)
__global__ void reciprocal_all(unsigned long long *count, uint32_t *first)
{
    const uint32_t lo = 0x0D800000u, n = 0x71800000u - 0x0D800000u;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float b = __uint_as_float(lo + i);
        const uint32_t got = __float_as_uint(reciprocal_rn(b)), want = __float_as_uint(__frcp_rn(b));
        // the pair form, b in the first lane, the range's mirror image in the second
        const float bo = __uint_as_float(lo + n - 1u - i);
        const float2 g2 = reciprocal_rn2(make_float2(b, bo), make_float2(-b, -bo));
        if (got != want || __float_as_uint(g2.x) != want ||
            __float_as_uint(g2.y) != __float_as_uint(__frcp_rn(bo)))
            note(count, first, lo + i, 0, got, want);
    }
}

// whole codes as the requantiser forms them (pairs of quotients, zeros as +0),
// against count_below(IEEE quotient)
__global__ void codes_random(const float *qmap, uint64_t n, uint64_t seed, unsigned long long *count,
                             uint32_t *first)
{
    __shared__ float q[256], mid[512];
    __shared__ uint8_t table[kBuckets];
    __shared__ uint32_t red[32];
    const int tid = threadIdx.x;
    q[tid] = qmap[tid];
    __syncthreads();
    mid[tid] = tid < 255 ? __fmul_rn(__fadd_rn(q[tid], q[tid + 1]), 0.5f) : INFINITY;
    mid[256 + tid] = INFINITY;
    __syncthreads();
    const int k = build_buckets(mid, table, red);
    __syncthreads();
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + tid; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t r0 = mix32(3 * i + seed), r1 = mix32(3 * i + 1 + seed), r2 = mix32(3 * i + 2 + seed);
        const uint32_t sb = 0x0D800000u + r0 % 0x64000000u;  // scale in the fast range
        const uint32_t drop = (r1 >> 24) % 160u;
        uint32_t xb = (r1 & 0x007FFFFFu) | ((sb & 0x7F800000u) - (drop << 23) * ((sb >> 23) > drop));
        if ((sb >> 23) <= drop) xb = r1 & 0x007FFFFFu;
        if (xb > sb) xb = sb;
        if ((r2 & 0xFFu) == 0u) xb = 0u;
        xb |= r2 & 0x80000000u;
        const float x = __uint_as_float(xb), s = __uint_as_float(sb);
        // the pair form, x beside a second value of the same block (|x'| <= scale)
        const float x2 = __uint_as_float((r2 >> 8) % (sb + 1u) | (r0 & 0x80000000u));
        const float2 c = divide_pair_for_code(make_float2(x, x2), make_float2(-s, -s),
                                              make_float2(reciprocal_rn(s), reciprocal_rn(s)));
        const float xs[2] = {x, x2}, cs[2] = {c.x, c.y};
        for (int j = 0; j < 2; ++j) {
            uint32_t got;
            if (fabsf(xs[j]) < __uint_as_float(fast_quotient_floor(sb)) &&
                needs_ieee_divide(xs[j], fast_quotient_floor(sb)))
                got = (uint32_t)count_below(mid, __fdiv_rn(xs[j], s));
            else
                got = k <= 2 ? code_by_bucket<2>(mid, table, cs[j], k) : code_by_bucket<0>(mid, table, cs[j], k);
            const uint32_t want = (uint32_t)count_below(mid, __fdiv_rn(xs[j], s));
            if (got != want)
                note(count, first, __float_as_uint(xs[j]), sb, got, want);
        }
    }
}

extern "C" int run_reciprocal_all(unsigned long long *count_host, uint32_t *first_host)
{
    unsigned long long *c; uint32_t *f;
    if (cudaMalloc(&c, 8) || cudaMalloc(&f, 16)) return -1;
    cudaMemset(c, 0, 8); cudaMemset(f, 0, 16);
    reciprocal_all<<<152 * 8, 256>>>(c, f);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(count_host, c, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(first_host, f, 16, cudaMemcpyDeviceToHost);
    cudaFree(c); cudaFree(f);
    return e;
}

extern "C" int run_codes_random(const float *qmap_host, uint64_t n, uint64_t seed,
                                unsigned long long *count_host, uint32_t *first_host)
{
    float *q; unsigned long long *c; uint32_t *f;
    if (cudaMalloc(&q, 256 * 4) || cudaMalloc(&c, 8) || cudaMalloc(&f, 16)) return -1;
    cudaMemcpy(q, qmap_host, 256 * 4, cudaMemcpyHostToDevice);
    cudaMemset(c, 0, 8); cudaMemset(f, 0, 16);
    codes_random<<<152 * 4, kThreadsPerBlockwiseCta>>>(q, n, seed, c, f);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(count_host, c, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(first_host, f, 16, cudaMemcpyDeviceToHost);
    cudaFree(q); cudaFree(c); cudaFree(f);
    return e;
}

extern "C" int run_divide_random(uint64_t n, uint64_t seed, unsigned long long *count_host, uint32_t *first_host)
{
    unsigned long long *c; uint32_t *f;
    if (cudaMalloc(&c, 8) || cudaMalloc(&f, 16)) return -1;
    cudaMemset(c, 0, 8); cudaMemset(f, 0, 16);
    divide_random<<<152 * 8, 256>>>(n, seed, c, f);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(count_host, c, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(first_host, f, 16, cudaMemcpyDeviceToHost);
    cudaFree(c); cudaFree(f);
    return e;
}
