// GPU checks of the staging primitives (test code): a bulk copy completes its
// mbarrier with the right bytes; an arrival completes a phase; a wait on a
// phase that nothing completes gives up after the bounded time and reports
// it, leaving the GPU usable.  One CTA of one thread per check.
#include <cuda_runtime.h>
#include <cstdint>
#include "pipeline.cuh"

using namespace pa;

// out[0]: 1 if the wait succeeded; out[1]: elapsed ns; out[2..]: copied words
__global__ void copy_check(const uint32_t *src, uint32_t nwords, uint64_t *out)
{
    __shared__ __align__(16) uint32_t buf[1024];
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    mbar_init_fence();
    const uint64_t t0 = global_ns();
    mbar_arrive_expect(&bar, nwords * 4u);
    bulk_load(buf, src, nwords * 4u, &bar);
    const bool ok = mbar_wait(&bar, 0);
    out[0] = ok ? 1u : 0u;
    out[1] = global_ns() - t0;
    for (uint32_t i = 0; i < nwords; ++i)
        out[2 + i] = ok ? buf[i] : 0xFFFFFFFFu;
}

// mode 0: arrive then wait (completes); mode 1: wait on a phase nobody completes
__global__ void wait_check(int mode, uint64_t *out)
{
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    mbar_init_fence();
    if (mode == 0)
        mbar_arrive(&bar);
    const uint64_t t0 = global_ns();
    const bool ok = mbar_wait(&bar, 0);
    out[0] = ok ? 1u : 0u;
    out[1] = global_ns() - t0;
}

extern "C" int run_copy_check(const uint32_t *src_host, uint32_t nwords, uint64_t *out_host)
{
    if (nwords == 0 || nwords > 1024 || nwords % 4 != 0) return -1;
    uint32_t *src; uint64_t *out;
    if (cudaMalloc(&src, nwords * 4) || cudaMalloc(&out, (2 + nwords) * 8)) return -1;
    cudaMemcpy(src, src_host, nwords * 4, cudaMemcpyHostToDevice);
    copy_check<<<1, 1>>>(src, nwords, out);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(out_host, out, (2 + nwords) * 8, cudaMemcpyDeviceToHost);
    cudaFree(src); cudaFree(out);
    return e;
}

extern "C" int run_wait_check(int mode, uint64_t *out_host)
{
    uint64_t *out;
    if (cudaMalloc(&out, 16)) return -1;
    wait_check<<<1, 1>>>(mode, out);
    const int e = (int)cudaDeviceSynchronize();
    cudaMemcpy(out_host, out, 16, cudaMemcpyDeviceToHost);
    cudaFree(out);
    return e;
}
