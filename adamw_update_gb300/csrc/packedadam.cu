// packedadam.cu -- CUDA kernels (sm_103a) and the C ABI of libpackedadam.so.
//
// The AdamW update with packed persistent moment state ("Packed AdamW
// Reference" README v1.0.0, "The canonical format"; "Packed AdamW / Reference
// / v1.0.0" code page, "Release scope"), its FP32 and FP16-first/FP16-RMS
// comparison modes, and the 8-bit blockwise mode of KBench
// "quantized-optimizer-state" reference.py (quantized_adamw_step,
// _requantise).  The declarations, numerics and error rules are documented in
// include/packedadam.h.
//
// Design.  The step is elementwise and bound by HBM bandwidth (20 bytes per
// parameter for the packed modes) and by instruction issue (the correctly
// rounded divisions and square roots, the codecs' integer work).  The
// consumers update 16-byte vectors four elements at a time with packed f32x2
// arithmetic, one warp vote choosing branch-free correctly rounded quotients
// and roots (exact.cuh) where every lane's operands allow them, the zero-safe
// IEEE arithmetic otherwise (codecs.cuh).  The step kernels are staged: one CTA
// per SM, whose producer warp streams tiles of every input into a two-stage
// shared-memory ring with bulk (TMA) copies and mbarriers, while 24 consumer
// warps update the staged tiles and store the results straight to global
// memory with streaming hints (adamw_step_pipe_kernel; blockwise8_pipe_kernel
// has 32 warps and no producer: the last warp to hand a stage back refills it).
// A multi-tensor list becomes one launch over a device-side descriptor table,
// whose tile prefix sums let the producer walk from tensor to tensor without a
// search; it hands each tile's geometry to the consumers with the tile.  The
// register-staged adamw_step_kernel (every thread issues its 16-byte loads
// before its arithmetic) serves the step on host-resident memory.  No tensor
// cores: nothing here is a contraction.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>
#include <vector>

#include "blockwise.cuh"
#include "codecs.cuh"
#include "packedadam.h"
#include "pipeline.cuh"

namespace pa {

// ---- the register-staged kernel (step on host memory) and the codecs ----------
constexpr int kThreads = 256;         // threads per CTA
#ifndef PA_UNROLL
#define PA_UNROLL 2
#endif
#ifndef PA_MIN_BLOCKS
#define PA_MIN_BLOCKS 4
#endif
constexpr int kUnroll = PA_UNROLL;    // 16-byte vectors per thread per chunk
// Resident CTAs per SM the step kernels are compiled for (caps registers at
// 65536 / (256 * 4) = 64): measured on GB300, 4 x 256 threads with two
// 16-byte vectors of each stream per thread beat 3 CTAs with four vectors by
// 19 %, the larger body also missing in the instruction cache.
constexpr int kMinBlocks = PA_MIN_BLOCKS;
#ifndef PA_NOALLOC_MAX_TENSORS
#define PA_NOALLOC_MAX_TENSORS 1024
#endif
constexpr int64_t kWave = (int64_t)kThreads * kUnroll * 4;  // elements per wave
constexpr int kMaxWaves = 8;  // waves per chunk, at most (chosen per launch)

enum Mode : int { kE4 = 0, kFP16 = 1, kF32 = 2 };

// One tensor of a step.  The 16-byte body starts `head` elements in; `vec`
// is 0 when p, g and the state do not share their address modulo 16, and the
// tensor then runs on 4-byte accesses.
struct Desc {
    float *p;
    const float *g;
    void *s1;        // uint32 words (packed modes) or FP32 m
    void *s2;        // FP32 v (FP32 mode)
    int64_t n;
    int64_t chunk0;  // first global work unit of this tensor: tile (staged kernels) or chunk
    int32_t head;
    int32_t vec;
};

// ---- memory access helpers --------------------------------------------------
__device__ __forceinline__ float4 load_stream(const float *a) { return __ldcs(reinterpret_cast<const float4 *>(a)); }
__device__ __forceinline__ uint4 load_stream(const uint32_t *a) { return __ldcs(reinterpret_cast<const uint4 *>(a)); }
__device__ __forceinline__ float4 load_readonly(const float *a) { return __ldg(reinterpret_cast<const float4 *>(a)); }
// four bfloat16 gradients (8 bytes) widened exactly to binary32
__device__ __forceinline__ float4 load_readonly(const __nv_bfloat16 *a)
{
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(a));
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
}
__device__ __forceinline__ float load_grad(const float *g, int64_t i) { return __ldg(g + i); }
__device__ __forceinline__ float load_grad(const __nv_bfloat16 *g, int64_t i)
{
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(g) + i) << 16);
}
__device__ __forceinline__ void store_stream(float *a, float4 x) { __stcs(reinterpret_cast<float4 *>(a), x); }
__device__ __forceinline__ void store_stream(uint32_t *a, uint4 x) { __stcs(reinterpret_cast<uint4 *>(a), x); }

// ---- one element of a packed step -------------------------------------------
// Decode the prior state, v = r*r, FP32 update, encode m' and sqrt(v') into the
// next word ("Release scope": the state is stored only after the update).
template <int MODE, bool UNIT_BC2>
__device__ __forceinline__ uint32_t packed_element(float &p, float g, uint32_t w,
                                                   const Scalars &s, uint32_t &bad)
{
    const float m = MODE == kE4 ? decode_m_lane(w) : decode_fp16_low(w);
    const float r = MODE == kE4 ? decode_rms_lane(w) : decode_fp16_high(w);
    float rn = 0.0f;
    const Moments o = adamw_element<UNIT_BC2>(p, g, m, __fmul_rn(r, r), s, &rn);
    bad += any_nonfinite(o);
    p = o.p;
    if (!UNIT_BC2)
        rn = __fsqrt_rn(o.v);  // bc2 == 1: the update took sqrt(v')
    return MODE == kE4 ? encode_step_word_e4(o.m, o.v, rn) : encode_word_fp16(o.m, rn);
}

// Four elements of packed_element (one staged vector) with packed arithmetic:
// the exact rebias multiplies of the E4 decode, v = r*r and the update's
// multiplies and adds one instruction per pair, the quotients and roots as
// adamw_vector chooses them for the warp; same bits.  Warp-collective.
__device__ __forceinline__ float2 decode_m_pair(uint32_t w0, uint32_t w1)
{
    const uint32_t b0 = ((w0 & 0x7FFFu) << 12) | ((w0 & 0x8000u) << 16);
    const uint32_t b1 = ((w1 & 0x7FFFu) << 12) | ((w1 & 0x8000u) << 16);
    return mul2(make_float2(__uint_as_float(b0), __uint_as_float(b1)), make_float2(0x1p112f, 0x1p112f));
}

__device__ __forceinline__ float2 decode_rms_pair(uint32_t w0, uint32_t w1)
{
    const uint32_t b0 = (w0 >> 5) & 0x07FFF800u, b1 = (w1 >> 5) & 0x07FFF800u;
    return mul2(make_float2(__uint_as_float(b0), __uint_as_float(b1)), make_float2(0x1p112f, 0x1p112f));
}

template <int MODE, bool UNIT_BC2, bool DEFER_NAN, bool PAIRED>
__device__ __forceinline__ uint4 packed_vector(float pp[4], const float gg[4], const uint4 w,
                                               const Scalars &s, const Pairs &k, const ZeroSafe &zs,
                                               uint32_t &bad)
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    float2 p[2], g[2], m[2], v[2], rn[2];
    Moments2 o[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        p[j] = make_float2(pp[2 * j], pp[2 * j + 1]);
        g[j] = make_float2(gg[2 * j], gg[2 * j + 1]);
        m[j] = MODE == kE4 ? decode_m_pair(ww[2 * j], ww[2 * j + 1])
                           : make_float2(decode_fp16_low(ww[2 * j]), decode_fp16_low(ww[2 * j + 1]));
        const float2 r = MODE == kE4 ? decode_rms_pair(ww[2 * j], ww[2 * j + 1])
                                     : make_float2(decode_fp16_high(ww[2 * j]), decode_fp16_high(ww[2 * j + 1]));
        v[j] = mul2(r, r);
    }
    adamw_vector<UNIT_BC2, true, PAIRED>(p, g, m, v, s, k, zs, o, rn);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        pp[2 * j] = o[j].p.x;
        pp[2 * j + 1] = o[j].p.y;
    }
    uint32_t out[4];
    // DEFER_NAN: encode without the NaN tests and only when the non-finite
    // count is nonzero encode again with them.  A NaN m' makes p' NaN and a
    // NaN RMS comes from a NaN v', so a lane whose code needs the NaN rules
    // always makes that count nonzero.  Same words either way.
    const uint32_t nf = DEFER_NAN ? 0u : nonfinite_count4(o);
    bad += nf;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (DEFER_NAN) {
            out[2 * j] = MODE == kE4 ? encode_step_word_e4_finite(o[j].m.x, rn[j].x)
                                     : encode_word_fp16_finite(o[j].m.x, rn[j].x);
            out[2 * j + 1] = MODE == kE4 ? encode_step_word_e4_finite(o[j].m.y, rn[j].y)
                                         : encode_word_fp16_finite(o[j].m.y, rn[j].y);
        } else {
            out[2 * j] = MODE == kE4 ? encode_step_word_e4(o[j].m.x, o[j].v.x, rn[j].x)
                                     : encode_word_fp16(o[j].m.x, rn[j].x);
            out[2 * j + 1] = MODE == kE4 ? encode_step_word_e4(o[j].m.y, o[j].v.y, rn[j].y)
                                         : encode_word_fp16(o[j].m.y, rn[j].y);
        }
    }
    if (DEFER_NAN) {
        const uint32_t nfd = nonfinite_count4(o);
        if (nfd != 0) {
            bad += nfd;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                out[2 * j] = MODE == kE4 ? encode_step_word_e4(o[j].m.x, o[j].v.x, rn[j].x)
                                         : encode_word_fp16(o[j].m.x, rn[j].x);
                out[2 * j + 1] = MODE == kE4 ? encode_step_word_e4(o[j].m.y, o[j].v.y, rn[j].y)
                                             : encode_word_fp16(o[j].m.y, rn[j].y);
            }
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Element i of tensor d with 4-byte accesses (heads, tails, unaligned tensors).
template <int MODE, bool U1, typename GT = float>
__device__ __forceinline__ void scalar_element(const Desc &d, int64_t i, const Scalars &s,
                                               uint32_t &bad)
{
    float p = d.p[i];
    const float g = load_grad(reinterpret_cast<const GT *>(d.g), i);
    if constexpr (MODE == kF32) {
        float *m = static_cast<float *>(d.s1);
        float *v = static_cast<float *>(d.s2);
        const Moments o = adamw_element<U1>(p, g, m[i], v[i], s);
        bad += any_nonfinite(o);
        d.p[i] = o.p;
        m[i] = o.m;
        v[i] = o.v;
    } else {
        uint32_t *w = static_cast<uint32_t *>(d.s1);
        const uint32_t nw = packed_element<MODE, U1>(p, g, w[i], s, bad);
        d.p[i] = p;
        w[i] = nw;
    }
}

// Chunk k of a 16-byte-path tensor: body elements [k*chunk, (k+1)*chunk)
// counted from d.head, walked as waves of kWave elements.  In a wave a
// thread issues all of its 16-byte loads (kUnroll vectors of p, g and the
// state) before any arithmetic; the per-thread pointers are set up once per
// chunk and advanced by a constant per wave.
template <int MODE, bool U1, typename GT = float>
__device__ __forceinline__ void vector_chunk(const Desc &d, int64_t k, int64_t chunk,
                                             const Scalars &s, uint32_t &bad)
{
    const int tid = threadIdx.x;
    const int64_t nb = d.n - d.head;
    int64_t base = k * chunk;
    if (k == 0 && tid < d.head)
        scalar_element<MODE, U1, GT>(d, tid, s, bad);
    const int64_t end = base + chunk < nb ? base + chunk : nb;
    const int64_t off = d.head + base + 4 * tid;
    float *P = d.p + off;
    const GT *G = reinterpret_cast<const GT *>(d.g) + off;
    uint32_t *W = static_cast<uint32_t *>(d.s1) + off;   // packed modes
    float *M = static_cast<float *>(d.s1) + off;         // FP32 mode
    float *V = static_cast<float *>(d.s2) + off;
    constexpr int kStride = kThreads * 4;  // elements between a thread's vectors
#pragma unroll 1
    for (; base < end; base += kWave, P += kWave, G += kWave, W += kWave, M += kWave, V += kWave) {
        const bool whole = base + kWave <= nb;  // uniform: no per-vector bound checks
        float4 pv[kUnroll], gv[kUnroll];
        uint4 wv[kUnroll];
        float4 mv[kUnroll], vv[kUnroll];
        bool full[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            full[u] = whole || base + 4 * ((int64_t)u * kThreads + tid) + 4 <= nb;
            if (full[u]) {
                pv[u] = load_stream(P + u * kStride);
                gv[u] = load_readonly(G + u * kStride);
                if constexpr (MODE == kF32) {
                    mv[u] = load_stream(M + u * kStride);
                    vv[u] = load_stream(V + u * kStride);
                } else {
                    wv[u] = load_stream(W + u * kStride);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (full[u]) {
                float pp[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
                const float gg[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
                if constexpr (MODE == kF32) {
                    float mm[4] = {mv[u].x, mv[u].y, mv[u].z, mv[u].w};
                    float vq[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const Moments o = adamw_element<U1>(pp[j], gg[j], mm[j], vq[j], s);
                        bad += any_nonfinite(o);
                        pp[j] = o.p;
                        mm[j] = o.m;
                        vq[j] = o.v;
                    }
                    store_stream(M + u * kStride, make_float4(mm[0], mm[1], mm[2], mm[3]));
                    store_stream(V + u * kStride, make_float4(vq[0], vq[1], vq[2], vq[3]));
                } else {
                    uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        ww[j] = packed_element<MODE, U1>(pp[j], gg[j], ww[j], s, bad);
                    store_stream(W + u * kStride, make_uint4(ww[0], ww[1], ww[2], ww[3]));
                }
                store_stream(P + u * kStride, make_float4(pp[0], pp[1], pp[2], pp[3]));
            } else {
                // the one vector that straddles the end of the tensor
                const int64_t e = base + 4 * ((int64_t)u * kThreads + tid);
                for (int64_t i = e; i < nb; ++i)
                    scalar_element<MODE, U1, GT>(d, d.head + i, s, bad);
            }
        }
    }
}

// Chunk k of a 4-byte-path tensor: elements [k*chunk, (k+1)*chunk).
template <int MODE, bool U1, typename GT = float>
__device__ __forceinline__ void scalar_chunk(const Desc &d, int64_t k, int64_t chunk,
                                             const Scalars &s, uint32_t &bad)
{
    const int64_t base = k * chunk;
    const int64_t end = base + chunk < d.n ? base + chunk : d.n;
#pragma unroll 4
    for (int64_t i = base + threadIdx.x; i < end; i += kThreads)
        scalar_element<MODE, U1, GT>(d, i, s, bad);
}

__device__ __forceinline__ void flush_nonfinite(uint32_t bad, unsigned long long *nonfinite)
{
    if (nonfinite == nullptr)
        return;
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bad);
    if ((threadIdx.x & 31) == 0 && total != 0)
        atomicAdd(nonfinite, (unsigned long long)total);
}

// The persistent step body.  MULTI: walk the device descriptor table (each
// CTA visits chunks in increasing order, so the tensor index only moves
// forward); otherwise the single descriptor passed by value.  U1: bc2 == 1.
template <int MODE, bool MULTI, bool U1, typename GT = float>
__device__ __forceinline__ void adamw_step_body(const Desc *__restrict__ table, int32_t ntensors,
                                                int64_t total_chunks, int64_t chunk,
                                                const Desc &single, const Scalars &s,
                                                unsigned long long *nonfinite)
{
    uint32_t bad = 0;
    int32_t t = 0;
    Desc d = single;
    int64_t next = total_chunks;
    if constexpr (MULTI) {
        d = table[0];
        next = ntensors > 1 ? table[1].chunk0 : total_chunks;
    }
    for (int64_t c = blockIdx.x; c < total_chunks; c += gridDim.x) {
        if constexpr (MULTI) {
            while (c >= next) {
                ++t;
                d = table[t];
                next = t + 1 < ntensors ? table[t + 1].chunk0 : total_chunks;
            }
        }
        const int64_t k = c - d.chunk0;
        if (d.vec)
            vector_chunk<MODE, U1, GT>(d, k, chunk, s, bad);
        else
            scalar_chunk<MODE, U1, GT>(d, k, chunk, s, bad);
    }
    flush_nonfinite(bad, nonfinite);
}

template <int MODE, bool MULTI, bool U1, typename GT = float>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
adamw_step_kernel(const Desc *__restrict__ table, int32_t ntensors, int64_t total_chunks,
                  int64_t chunk, const Desc single, const Scalars s,
                  unsigned long long *nonfinite)
{
    adamw_step_body<MODE, MULTI, U1, GT>(table, ntensors, total_chunks, chunk, single, s,
                                         nonfinite);
}

// ---- the staged step (FP32 or bfloat16 gradients) -----------------------------
// One CTA per SM: a producer warp whose lane 0 streams tiles of p, g and the
// state (p, g, m, v in the FP32 mode) into a two-stage shared-memory ring
// with bulk (TMA) copies, and 24 consumer warps that update a staged tile
// from shared memory and store p' and the new state straight to global memory
// with streaming hints.  The copies of the next tile are in flight while the
// consumers work on the current one, so HBM sees a steady stream of large
// reads without the registers that register-staged loads would hold, and the
// 768 consumer threads have enough independent elements (8 each per tile) to
// hide the latency of the division and square-root chains.  Measured on
// GB300 (10^9 parameters, packed E4): 6144-element tiles with 24 consumer
// warps and two stages ran at 1.13x the register-staged kernel; 8 consumer
// warps could not keep up with the copies.
//
// A tile covers kTile elements of one tensor's 16-byte body (from d.head on);
// the last tile of a tensor may be shorter: its largest multiple of four
// elements is copied and the remaining <= 3, like the <= 3 head elements, are
// updated from global memory by single consumer threads.  A tensor on the
// 4-byte path (streams not sharing their address modulo 16) is cut into
// tiles the same way but updated from global memory, with no copies.
constexpr int kTile = 6144;
constexpr int kStages = 2;
constexpr int kConsumerWarps = 24;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kPipeThreads = kConsumers + 32;  // + the producer warp
constexpr int kTileVecs = kTile / (4 * kConsumers);
static_assert(kTile % (4 * kConsumers) == 0, "a tile is whole 16-byte vectors per consumer");
static_assert(sizeof(Desc) % sizeof(uint64_t) == 0, "descriptors copy as 8-byte words");

// Lists of up to kSmemDescs tensors have their descriptor table copied into
// shared memory at kernel start, so the producer's walk from tensor to tensor
// costs no dependent global loads (with tens of tensors and few tiles each,
// those loads outlasted a tile's computation).
constexpr int kSmemDescs = 512;

// What the consumers need to know about a staged tile, written by the
// producer into the stage's slot before it signals the stage, so that only
// the producer walks the descriptor table.
struct TileInfo {
    float *p;
    const void *g;
    void *s1, *s2;
    int64_t base;     // first element of the tile in its tensor
    int32_t len;      // elements in the tile
    int32_t staged;   // of them, staged by the bulk copies
    int32_t head;     // elements before the 16-byte body, updated with this tile
    int32_t vec;      // the tensor's body is staged (else 4-byte accesses)
};

// A stage holds one tile of each stream: p, g (GT: float or bfloat16), the
// state word or m, and v in the FP32 mode; after the stages come the
// barriers and the shared copy of the descriptor table.
template <int MODE, typename GT = float>
struct PipeLayout {
    static constexpr size_t kG = (size_t)kTile * 4;                 // gradients
    static constexpr size_t kS1 = kG + (size_t)kTile * sizeof(GT);  // state word | m
    static constexpr size_t kS2 = kS1 + (size_t)kTile * 4;          // v (FP32 mode)
    static constexpr size_t kStageBytes = MODE == kF32 ? kS2 + (size_t)kTile * 4 : kS2;
    static constexpr size_t kBarriers = kStages * kStageBytes;
    static constexpr size_t kInfo = kBarriers + 2 * kStages * sizeof(uint64_t);
    static constexpr size_t kDescs = kInfo + kStages * sizeof(TileInfo);
    static constexpr size_t kBytes = kDescs + (size_t)kSmemDescs * sizeof(Desc);  // the most
    // dynamic shared memory of a launch over `ntensors` tensors
    static size_t bytes_for(int32_t ntensors)
    {
        return kDescs + (ntensors <= kSmemDescs ? (size_t)ntensors * sizeof(Desc) : 0);
    }
    static constexpr uint32_t kBytesPerElem = (uint32_t)(kStageBytes / kTile);
    // a staged run is whole 16-byte units of every stream: 4 elements, 8 for bfloat16
    static constexpr int kUnit = sizeof(GT) == 2 ? 8 : 4;
};

// Set (first code wins) when a bounded wait of a staged kernel gives up; the
// launch's results are then incomplete.  Read and cleared by pa_device_fault.
enum PipeFault : uint32_t {
    kFaultEmptyWait = 1,  // the producer waited > 2 s for consumers to free a stage
    kFaultCopyWait = 2,   // the producer waited > 2 s for its last copies to land
    kFaultFullWait = 3,   // a consumer waited > 2 s for a stage's copies
};
static __device__ uint32_t g_pipe_fault;

__device__ __forceinline__ void pipe_fault(uint32_t code)
{
    atomicCAS(&g_pipe_fault, 0u, code);
}

// Elements [base, base + len) of the tensor form tile k; the first `staged`
// of them (whole units of `unit` elements: 4, or 8 with bfloat16 gradients)
// are staged by bulk copies (none on the 4-byte path).
struct Span {
    int64_t base;
    int32_t len, staged;
};

__device__ __forceinline__ Span tile_span(const Desc &d, int64_t k, int unit, int32_t tile)
{
    const int64_t b = k * tile;
    int64_t len = (d.vec ? d.n - d.head : d.n) - b;
    len = len < 0 ? 0 : (len > tile ? tile : len);
    Span sp;
    sp.base = d.vec ? d.head + b : b;
    sp.len = (int32_t)len;
    sp.staged = d.vec ? (int32_t)(len & ~(int64_t)(unit - 1)) : 0;
    return sp;
}

// Walks the descriptor table forward to the tensor of global tile c.
struct TableCursor {
    const Desc *table;
    int32_t ntensors, t;
    int64_t next;
    Desc d;
    __device__ __forceinline__ TableCursor(const Desc *tab, int32_t nt, int64_t total)
        : table(tab), ntensors(nt), t(0), next(nt > 1 ? tab[1].chunk0 : total), d(tab[0])
    {
    }
    __device__ __forceinline__ void seek(int64_t c, int64_t total)
    {
        while (c >= next) {
            ++t;
            d = table[t];
            next = t + 1 < ntensors ? table[t + 1].chunk0 : total;
        }
    }
};

template <int MODE, typename GT>
__device__ __forceinline__ void pipe_produce(unsigned char *smem, uint64_t *full, uint64_t *empty,
                                             const Desc *table, int32_t ntensors, int64_t total,
                                             int32_t tile)
{
    using L = PipeLayout<MODE, GT>;
    TileInfo *info = reinterpret_cast<TileInfo *>(smem + L::kInfo);
    TableCursor cur(table, ntensors, total);
    int64_t k = 0;  // fills issued
    for (int64_t c = blockIdx.x; c < total; c += gridDim.x, ++k) {
        cur.seek(c, total);
        const int st = (int)(k % kStages);
        const uint32_t use = (uint32_t)(k / kStages);
        if (!mbar_wait(&empty[st], (use & 1u) ^ 1u)) {  // the first use passes at once
            pipe_fault(kFaultEmptyWait);
            break;
        }
        const int64_t kt = c - cur.d.chunk0;
        const Span sp = tile_span(cur.d, kt, L::kUnit, tile);
        TileInfo &ti = info[st];
        ti.p = cur.d.p;
        ti.g = cur.d.g;
        ti.s1 = cur.d.s1;
        ti.s2 = cur.d.s2;
        ti.base = sp.base;
        ti.len = sp.len;
        ti.staged = sp.staged;
        ti.head = (cur.d.vec && kt == 0) ? cur.d.head : 0;
        ti.vec = cur.d.vec;
        const uint32_t units = (uint32_t)sp.staged;
        mbar_arrive_expect(&full[st], units * L::kBytesPerElem);  // releases the slot too
        if (units != 0) {
            unsigned char *buf = smem + (size_t)st * L::kStageBytes;
            bulk_load(buf, cur.d.p + sp.base, units * 4u, &full[st]);
            bulk_load(buf + L::kG, reinterpret_cast<const GT *>(cur.d.g) + sp.base,
                      units * (uint32_t)sizeof(GT), &full[st]);
            bulk_load(buf + L::kS1, static_cast<const uint32_t *>(cur.d.s1) + sp.base, units * 4u,
                      &full[st]);
            if (MODE == kF32)
                bulk_load(buf + L::kS2, static_cast<const float *>(cur.d.s2) + sp.base, units * 4u,
                          &full[st]);
        }
    }
    // The CTA's shared memory must outlive its copies: wait for the last fill
    // of every stage before leaving.
    for (int64_t j = k > kStages ? k - kStages : 0; j < k; ++j)
        if (!mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1)))
            pipe_fault(kFaultCopyWait);
}

// One staged 16-byte vector: elements e..e+3 of the stage buffer, which are
// elements base+e.. of the tensor (warp-collective: adamw_vector).  PAIRED:
// the branch-free arm in packed pairs (these vectors are issue-bound: 2.7 %
// faster on gpt2-148; the graph-replayable kernel, which holds its scalars in
// registers, spilled with it and keeps the scalar arm).
template <int MODE, bool U1, typename GT, bool PAIRED>
__device__ __forceinline__ void pipe_vector_math(const unsigned char *buf, int e, const Desc &d,
                                                 int64_t base, float pp[4], const float gg[4],
                                                 const Scalars &s, const ZeroSafe &zs,
                                                 uint32_t &bad)
{
    using L = PipeLayout<MODE, GT>;
    const Pairs k = pairs_of(s);
    if constexpr (MODE == kF32) {
        const float4 mv = *reinterpret_cast<const float4 *>(buf + L::kS1 + 4 * e);
        const float4 vv = *reinterpret_cast<const float4 *>(buf + L::kS2 + 4 * e);
        const float2 p[2] = {make_float2(pp[0], pp[1]), make_float2(pp[2], pp[3])};
        const float2 g[2] = {make_float2(gg[0], gg[1]), make_float2(gg[2], gg[3])};
        const float2 m[2] = {make_float2(mv.x, mv.y), make_float2(mv.z, mv.w)};
        const float2 v[2] = {make_float2(vv.x, vv.y), make_float2(vv.z, vv.w)};
        Moments2 o[2];
        float2 unused[2];
        adamw_vector<U1, false, PAIRED>(p, g, m, v, s, k, zs, o, unused);
        bad += nonfinite_count4(o);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pp[2 * j] = o[j].p.x;
            pp[2 * j + 1] = o[j].p.y;
        }
        store_stream(static_cast<float *>(d.s1) + base + e, make_float4(o[0].m.x, o[0].m.y, o[1].m.x, o[1].m.y));
        store_stream(static_cast<float *>(d.s2) + base + e, make_float4(o[0].v.x, o[0].v.y, o[1].v.x, o[1].v.y));
    } else {
        const uint4 wv = *reinterpret_cast<const uint4 *>(buf + L::kS1 + 4 * e);
        // (the E4 vectors here are issue-bound: NaN tests deferred, 2 % faster
        // on gpt2-148; the FP16 mode measured no gain)
        store_stream(static_cast<uint32_t *>(d.s1) + base + e,
                     packed_vector<MODE, U1, MODE == kE4, PAIRED>(pp, gg, wv, s, k, zs, bad));
    }
}

// One staged vector whose gradients gv are already loaded.
template <int MODE, bool U1, typename GT, bool PAIRED>
__device__ __forceinline__ void pipe_vector_g(const unsigned char *buf, int e, const Desc &d,
                                              int64_t base, const float4 gv, const Scalars &s,
                                              const ZeroSafe &zs, uint32_t &bad)
{
    const float4 pv = *reinterpret_cast<const float4 *>(buf + 4 * e);
    float pp[4] = {pv.x, pv.y, pv.z, pv.w};
    const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
    pipe_vector_math<MODE, U1, GT, PAIRED>(buf, e, d, base, pp, gg, s, zs, bad);
    store_stream(d.p + base + e, make_float4(pp[0], pp[1], pp[2], pp[3]));
}

// One staged vector held in registers (the whole-tile path copies all of a
// thread's vectors out of the stage, hands the stage back, then computes).
template <int MODE>
struct RegVec {
    float4 p, g;
    uint4 w;      // packed modes
    float4 m, v;  // FP32 mode
};

template <int MODE, typename GT>
__device__ __forceinline__ RegVec<MODE> load_vec(const unsigned char *buf, int e, float4 g)
{
    using L = PipeLayout<MODE, GT>;
    RegVec<MODE> r;
    r.p = *reinterpret_cast<const float4 *>(buf + 4 * e);
    r.g = g;
    if constexpr (MODE == kF32) {
        r.m = *reinterpret_cast<const float4 *>(buf + L::kS1 + 4 * e);
        r.v = *reinterpret_cast<const float4 *>(buf + L::kS2 + 4 * e);
    } else {
        r.w = *reinterpret_cast<const uint4 *>(buf + L::kS1 + 4 * e);
    }
    return r;
}

// Every mode takes adamw_vector here (packed pairs, the warp's vote for the
// branch-free quotients and roots).  Measured on GB300 against one element at
// a time with the IEEE arithmetic: FP32 3 % faster on the gpt-52 list; packed
// E4 +0.2 % on the 7e9-parameter flat workload and +2.2 % with bfloat16
// gradients (that step is issue-bound), once the roots took their zero case
// by an add and the non-finite count went to packed FMAs (before that, 2.6 %
// slower on the flat workload).
template <int MODE, bool U1, typename GT, bool PAIRED>
__device__ __forceinline__ void compute_vec(const RegVec<MODE> &r, int e, const Desc &d,
                                            int64_t base, const Scalars &s, const ZeroSafe &zs,
                                            uint32_t &bad)
{
    float pp[4] = {r.p.x, r.p.y, r.p.z, r.p.w};
    const float gg[4] = {r.g.x, r.g.y, r.g.z, r.g.w};
    if constexpr (MODE == kF32) {
        const float2 p[2] = {make_float2(pp[0], pp[1]), make_float2(pp[2], pp[3])};
        const float2 g[2] = {make_float2(gg[0], gg[1]), make_float2(gg[2], gg[3])};
        const float2 m[2] = {make_float2(r.m.x, r.m.y), make_float2(r.m.z, r.m.w)};
        const float2 v[2] = {make_float2(r.v.x, r.v.y), make_float2(r.v.z, r.v.w)};
        Moments2 o[2];
        float2 unused[2];
        adamw_vector<U1, false, PAIRED>(p, g, m, v, s, pairs_of(s), zs, o, unused);
        bad += nonfinite_count4(o);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pp[2 * j] = o[j].p.x;
            pp[2 * j + 1] = o[j].p.y;
        }
        store_stream(static_cast<float *>(d.s1) + base + e, make_float4(o[0].m.x, o[0].m.y, o[1].m.x, o[1].m.y));
        store_stream(static_cast<float *>(d.s2) + base + e, make_float4(o[0].v.x, o[0].v.y, o[1].v.x, o[1].v.y));
    } else {
        // (NaN tests deferred and the branch-free arm in packed pairs with
        // bfloat16 gradients, whose whole tiles are issue-bound: 4 % and 6 %
        // faster; with FP32 gradients, bound by HBM, each measured 3-5 %
        // slower on the flat workload)
        store_stream(static_cast<uint32_t *>(d.s1) + base + e,
                     packed_vector<MODE, U1, sizeof(GT) == 2, PAIRED || sizeof(GT) == 2>(
                         pp, gg, r.w, s, pairs_of(s), zs, bad));
    }
    store_stream(d.p + base + e, make_float4(pp[0], pp[1], pp[2], pp[3]));
}

__device__ __forceinline__ bool has_zero(const float4 g)
{
    return g.x == 0.0f || g.y == 0.0f || g.z == 0.0f || g.w == 0.0f;
}

// four staged gradients as binary32 (bfloat16 widened exactly)
template <typename GT>
__device__ __forceinline__ float4 staged_grad(const unsigned char *buf, int e)
{
    if constexpr (sizeof(GT) == 2) {
        const uint2 r = *reinterpret_cast<const uint2 *>(buf + kTile * 4 + 2 * e);
        return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                           __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
    } else {
        return *reinterpret_cast<const float4 *>(buf + kTile * 4 + 4 * e);
    }
}

// Elements first, first+stride, ... below end, from global memory (head,
// ragged tail, 4-byte-path tensors).  (Inlined: as an out-of-line call it
// cost 2-9 % on GB300, the descriptor then living on the stack.)
template <int MODE, bool U1, typename GT>
__device__ __forceinline__ uint32_t pipe_scalar_run(const Desc &d, int64_t first, int64_t end,
                                                 int32_t stride, const Scalars &s)
{
    uint32_t bad = 0;
    for (int64_t i = first; i < end; i += stride)
        scalar_element<MODE, U1, GT>(d, i, s, bad);
    return bad;
}

// PAIR: 0 the branch-free arithmetic one lane at a time everywhere; 1 in
// packed pairs on the per-vector path (and, as always, with bfloat16
// gradients); 2 in packed pairs on the whole tiles too.
template <int MODE, bool U1, typename GT, int PAIR>
__device__ __forceinline__ void pipe_consume(const unsigned char *smem, uint64_t *full,
                                             uint64_t *empty, int64_t total, const Scalars &s,
                                             uint32_t &bad)
{
    using L = PipeLayout<MODE, GT>;
    const int ct = threadIdx.x;  // consumer thread, 0 .. kConsumers-1
    const ZeroSafe zs = zero_safe_of(s);
    const TileInfo *info = reinterpret_cast<const TileInfo *>(smem + L::kInfo);
    int64_t k = 0;
    for (int64_t c = blockIdx.x; c < total; c += gridDim.x, ++k) {
        const int st = (int)(k % kStages);
        if (!mbar_wait(&full[st], (uint32_t)((k / kStages) & 1))) {
            pipe_fault(kFaultFullWait);
            break;
        }
        const TileInfo ti = info[st];
        Desc d;
        d.p = ti.p;
        d.g = static_cast<const float *>(ti.g);
        d.s1 = ti.s1;
        d.s2 = ti.s2;
        d.vec = ti.vec;
        Span sp;
        sp.base = ti.base;
        sp.len = ti.len;
        sp.staged = ti.staged;
        const int32_t head_n = ti.head;
        bool released = false;
        if (d.vec) {
            const unsigned char *buf = smem + (size_t)st * L::kStageBytes;
            // Whole tile without a zero gradient in this warp: every vector
            // on the plain path, unrolled.  Otherwise one vector at a time,
            // each warp-vector choosing the branch-free or the zero-safe
            // arithmetic (adamw_vector; one copy of each: the E4 element is
            // large, and more inlined copies missed in the instruction cache
            // on GB300).  (Whole tiles of a runtime size below kTile, with the
            // vectors past the tile's end skipped, measured 3-9 % slower on
            // GB300 everywhere, also at kTile.)
            bool fast = sp.staged == kTile;  // uniform over the CTA
            float4 gv[kTileVecs];
            if (fast) {
                bool z = false;
#pragma unroll
                for (int v = 0; v < kTileVecs; ++v) {
                    gv[v] = staged_grad<GT>(buf, 4 * (ct + v * kConsumers));
                    z = z || has_zero(gv[v]);
                }
                fast = !__any_sync(0xFFFFFFFFu, z);
            }
            if (fast && MODE != kFP16) {
                // everything into registers, the stage back to the producer, then
                // compute (measured on GB300: +0.2 % E4, +0.4 % FP32, but -9 % in
                // the FP16 mode, which keeps the plain order below)
                RegVec<MODE> rv[kTileVecs];
#pragma unroll
                for (int v = 0; v < kTileVecs; ++v)
                    rv[v] = load_vec<MODE, GT>(buf, 4 * (ct + v * kConsumers), gv[v]);
                __syncwarp();
                if ((ct & 31) == 0)
                    mbar_arrive(&empty[st]);
                released = true;
#pragma unroll
                for (int v = 0; v < kTileVecs; ++v)
                    compute_vec<MODE, U1, GT, PAIR == 2>(rv[v], 4 * (ct + v * kConsumers), d, sp.base,
                                                         s, zs, bad);
            } else if (fast) {
#pragma unroll
                for (int v = 0; v < kTileVecs; ++v)
                    pipe_vector_g<MODE, U1, GT, (PAIR >= 1)>(buf, 4 * (ct + v * kConsumers), d, sp.base,
                                                gv[v], s, zs, bad);
            } else {
#pragma unroll 1
                for (int v = 0; v < kTileVecs; ++v) {
                    const int e = 4 * (ct + v * kConsumers);
                    if (e < sp.staged)
                        pipe_vector_g<MODE, U1, GT, (PAIR >= 1)>(buf, e, d, sp.base, staged_grad<GT>(buf, e), s,
                                                    zs, bad);
                }
            }
            // the <= 3 elements before the 16-byte body (first tile) and the
            // < unit after the staged part (last tile), one per thread
            const bool head = ct < head_n, tail = ct < sp.len - sp.staged;
            if (head || tail) {
#pragma unroll 1
                for (int r = head ? 0 : 1; r < (tail ? 2 : 1); ++r)
                    bad += pipe_scalar_run<MODE, U1, GT>(d, r == 0 ? ct : sp.base + sp.staged + ct,
                                                         (r == 0 ? ct : sp.base + sp.staged + ct) + 1,
                                                         1, s);
            }
        } else {
            bad += pipe_scalar_run<MODE, U1, GT>(d, sp.base + ct, sp.base + sp.len, kConsumers, s);
        }
        if (!released) {
            __syncwarp();
            if ((ct & 31) == 0)
                mbar_arrive(&empty[st]);
        }
    }
}

// table == nullptr: one tensor, described by `single` (ntensors == 1).  `tile`:
// elements per tile (kTile, or fewer for a launch too small to fill the GPU).
template <int MODE, bool U1, typename GT = float, int PAIR = 1>
__device__ __forceinline__ void pipe_body(const Desc *__restrict__ table, int32_t ntensors,
                                          int64_t total_tiles, const Desc &single,
                                          const Scalars &s, unsigned long long *nonfinite,
                                          int32_t tile)
{
    using L = PipeLayout<MODE, GT>;
    extern __shared__ __align__(128) unsigned char pipe_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(pipe_smem + L::kBarriers);
    uint64_t *empty = full + kStages;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init_fence();
    }
    // the producer's copy of the table, in 8-byte words, by every thread (one
    // or two loads each, so the first copies are not held up); a descriptor
    // passed by value is stored by thread 0.  (One tensor through this table
    // path measured 0.4 % faster on GB300 than a producer reading the
    // descriptor from the launch parameters.)
    const bool table_shared = ntensors <= kSmemDescs;
    if (table == nullptr) {
        if (threadIdx.x == 0)
            *reinterpret_cast<Desc *>(pipe_smem + L::kDescs) = single;
    } else if (table_shared) {
        const uint64_t *src = reinterpret_cast<const uint64_t *>(table);
        uint64_t *dst = reinterpret_cast<uint64_t *>(pipe_smem + L::kDescs);
        constexpr int kWords = sizeof(Desc) / sizeof(uint64_t);
        for (int i = threadIdx.x; i < ntensors * kWords; i += kPipeThreads)
            dst[i] = __ldg(src + i);
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers) {  // the producer warp
        if (table_shared)
            table = reinterpret_cast<const Desc *>(pipe_smem + L::kDescs);
        if (threadIdx.x == kConsumers)
            pipe_produce<MODE, GT>(pipe_smem, full, empty, table, ntensors, total_tiles, tile);
        return;
    }
    uint32_t bad = 0;
    pipe_consume<MODE, U1, GT, PAIR>(pipe_smem, full, empty, total_tiles, s, bad);
    flush_nonfinite(bad, nonfinite);
}

template <int MODE, bool U1, typename GT = float, int PAIR = 1>
__global__ void __launch_bounds__(kPipeThreads, 1)
adamw_step_pipe_kernel(const Desc *__restrict__ table, int32_t ntensors, int64_t total_tiles,
                       const Desc single, const Scalars s, unsigned long long *nonfinite,
                       int32_t tile)
{
    pipe_body<MODE, U1, GT, PAIR>(table, ntensors, total_tiles, single, s, nonfinite, tile);
}

// Graph-replayable variant: the scalars of the step are row *index of a
// device table filled by the host ahead of time, so a captured launch needs no
// host work per step.  An index outside [0, rows) sets *status to 1 and
// skips the update (nothing is written).
template <int MODE>
__global__ void __launch_bounds__(kPipeThreads, 1)
adamw_step_table_kernel(const Desc *__restrict__ table, int32_t ntensors, int64_t total_tiles,
                        const Scalars *__restrict__ rows, int32_t nrows,
                        const int64_t *__restrict__ index, int32_t *status,
                        unsigned long long *nonfinite)
{
    const int64_t i = *index;
    if (i < 0 || i >= nrows) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && status != nullptr)
            *status = 1;
        return;
    }
    const Scalars s = rows[i];
    Desc none = {};
    pipe_body<MODE, false, float, 0>(table, ntensors, total_tiles, none, s, nonfinite, kTile);
}

__global__ void advance_index_kernel(int64_t *index)
{
    *index += 1;
}

// ---- standalone codecs ("Packed AdamW Reference" README: inspect-formats) -------
template <int MODE>
__global__ void __launch_bounds__(kThreads)
encode_state_kernel(const float *__restrict__ m, const float *__restrict__ rms,
                    uint32_t *__restrict__ word, int64_t n, unsigned long long *nonfinite)
{
    uint32_t bad = 0;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        const float a = __ldg(m + i), b = __ldg(rms + i);
        word[i] = MODE == kE4 ? encode_word_e4(a, b) : encode_word_fp16(a, b);
        const uint32_t ea = __float_as_uint(a) & 0x7FFFFFFFu, eb = __float_as_uint(b) & 0x7FFFFFFFu;
        bad += max(ea, eb) >= 0x7F800000u ? 1u : 0u;
    }
    flush_nonfinite(bad, nonfinite);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads)
decode_state_kernel(const uint32_t *__restrict__ word, float *__restrict__ m,
                    float *__restrict__ rms, int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        const uint32_t w = __ldg(word + i);
        m[i] = MODE == kE4 ? decode_m_lane(w) : decode_fp16_low(w);
        rms[i] = MODE == kE4 ? decode_rms_lane(w) : decode_fp16_high(w);
    }
}

// Vectorised codecs: when m, rms and the words share their address modulo 16,
// the elements after the first `head` (< 4) go as 16-byte vectors, kUnroll of
// each array per thread and wave, every load of a wave issued before any
// arithmetic (the scalar kernels above keep one 4-byte load per thread in
// flight and wait on memory).  The head and the < 4 elements after the last
// whole vector are coded by single threads of the first CTA.
template <int MODE>
__global__ void __launch_bounds__(kThreads)
encode_state_vec_kernel(const float *__restrict__ m, const float *__restrict__ rms,
                        uint32_t *__restrict__ word, int64_t n, int64_t head,
                        unsigned long long *nonfinite)
{
    uint32_t bad = 0;
    const int64_t nv = (n - head) / 4;
    const float *M = m + head, *R = rms + head;
    uint32_t *W = word + head;
    const int64_t wave = (int64_t)gridDim.x * kThreads * kUnroll;
    for (int64_t v0 = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; v0 < nv; v0 += wave) {
        float4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < nv) {
                a[u] = load_stream(M + 4 * v);
                b[u] = load_stream(R + 4 * v);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < nv) {
                const float x[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
                const float y[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    w[j] = MODE == kE4 ? encode_word_e4(x[j], y[j]) : encode_word_fp16(x[j], y[j]);
                    const uint32_t ea = __float_as_uint(x[j]) & 0x7FFFFFFFu;
                    const uint32_t eb = __float_as_uint(y[j]) & 0x7FFFFFFFu;
                    bad += max(ea, eb) >= 0x7F800000u ? 1u : 0u;
                }
                store_stream(W + 4 * v, make_uint4(w[0], w[1], w[2], w[3]));
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 8) {  // head (threads 0..3) and tail (4..7)
        const int64_t i = threadIdx.x < 4 ? (int64_t)threadIdx.x : head + 4 * nv + threadIdx.x - 4;
        if ((threadIdx.x < 4 ? i < head : i < n)) {
            const float a = m[i], b = rms[i];
            word[i] = MODE == kE4 ? encode_word_e4(a, b) : encode_word_fp16(a, b);
            const uint32_t ea = __float_as_uint(a) & 0x7FFFFFFFu, eb = __float_as_uint(b) & 0x7FFFFFFFu;
            bad += max(ea, eb) >= 0x7F800000u ? 1u : 0u;
        }
    }
    flush_nonfinite(bad, nonfinite);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads)
decode_state_vec_kernel(const uint32_t *__restrict__ word, float *__restrict__ m,
                        float *__restrict__ rms, int64_t n, int64_t head)
{
    const int64_t nv = (n - head) / 4;
    const uint32_t *W = word + head;
    float *M = m + head, *R = rms + head;
    const int64_t wave = (int64_t)gridDim.x * kThreads * kUnroll;
    for (int64_t v0 = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; v0 < nv; v0 += wave) {
        uint4 a[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < nv)
                a[u] = load_stream(W + 4 * v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            if (v < nv) {
                const uint32_t w[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
                float x[4], y[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[j] = MODE == kE4 ? decode_m_lane(w[j]) : decode_fp16_low(w[j]);
                    y[j] = MODE == kE4 ? decode_rms_lane(w[j]) : decode_fp16_high(w[j]);
                }
                store_stream(M + 4 * v, make_float4(x[0], x[1], x[2], x[3]));
                store_stream(R + 4 * v, make_float4(y[0], y[1], y[2], y[3]));
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 8) {
        const int64_t i = threadIdx.x < 4 ? (int64_t)threadIdx.x : head + 4 * nv + threadIdx.x - 4;
        if ((threadIdx.x < 4 ? i < head : i < n)) {
            const uint32_t w = word[i];
            m[i] = MODE == kE4 ? decode_m_lane(w) : decode_fp16_low(w);
            rms[i] = MODE == kE4 ? decode_rms_lane(w) : decode_fp16_high(w);
        }
    }
}

// ---- 8-bit blockwise mode (KBench quantized_adamw_step, _requantise) -------------
// One CTA of 32 warps per SM (blockwise8_pipe_kernel below): a tile of four
// 2048-element blocks is bulk-copied into a two-stage shared-memory ring, and
// each group of 8 warps (256 threads) updates one block of the tile.  Thread t
// of a group holds elements 4t..4t+3 and 1024+4t..1024+4t+3 of its block.  The
// new block absmax is a warp max (redux.sync on the binary32 bits of |x|,
// which orders non-negative floats and lets a NaN win) followed by a max over
// the group's 8 warp results in shared memory at the group's named barrier.
//
// Requantisation, per element: c = x / max(absmax, 1e-30) and code = the
// number of the map's 255 midpoints strictly below c.
//  * Division.  When the block scale is a normal number in [2^-100, 2^100),
//    each thread takes y = RN(1/scale) once per block (reciprocal_rn: the
//    hardware approximation refined by one Newton-Raphson step, equal to the
//    IEEE reciprocal on that range) and forms c = RN(q0 + r*y) with
//    q0 = RN(x*y) and r = x - scale*q0 (exact by FMA): Markstein's theorem
//    (P. Markstein, IBM J. Res. Dev. 34(1), 1990) makes this the correctly
//    rounded quotient when y is the correctly rounded reciprocal and nothing
//    under- or overflows; here |x| <= scale, so that holds for |x| above a
//    floor; a zero x gives +0, whose code is that of -0; other nonzero |x|
//    below the floor use the IEEE divide in a rarely entered fix-up.  Two
//    values at a time, with packed arithmetic.
//  * Search.  A per-CTA table indexed by the top 14 bits of c's binary32
//    pattern (32 buckets per binade, either sign) holds the number of
//    midpoints below every value of the bucket; the code is that count plus K
//    comparisons with the following midpoints, K the largest number of
//    midpoints in one bucket (uniform over the CTA, so no divergence) -- exact
//    for any ascending map; K = 1 for the log-linear maps.
//  * A block whose scale is NaN, infinite or outside [2^-100, 2^100) takes
//    the IEEE divide and an 8-step binary search over the midpoints.
// Rare path: requantise a thread's 8 values with the IEEE divide and the
// binary search (block scale NaN, infinite or outside [2^-100, 2^100)).  Out
// of line to keep the hot loop's code small.
__device__ __noinline__ uint2 requantise_slow(float x0, float x1, float x2, float x3, float x4,
                                              float x5, float x6, float x7, float scale,
                                              const float *mid)
{
    const float x[8] = {x0, x1, x2, x3, x4, x5, x6, x7};
    uint2 code = make_uint2(0u, 0u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        code.x |= (uint32_t)count_below(mid, __fdiv_rn(x[j], scale)) << (8 * j);
        code.y |= (uint32_t)count_below(mid, __fdiv_rn(x[4 + j], scale)) << (8 * j);
    }
    return code;
}

struct BlockwiseArgs {
    const float *p;
    const float *g;
    uint16_t *p_bf16;
    uint8_t *m_code;
    float *m_absmax;
    uint8_t *v_code;
    float *v_absmax;
    int64_t n;
};

// Staged blockwise kernel: one CTA per SM; a tile is kBwGroups consecutive
// 2048-element blocks of one tensor, and consumer group j (8 warps, 256
// threads) updates block j of a tile.  32 warps (64 registers each) ran 1.2 %
// faster on GB300 than 24 warps with 80 registers.
constexpr int kBwWarps = 32;
constexpr int kBwThreads = kBwWarps * 32;
constexpr int kBwGroups = kBwWarps / 8;      // 4
constexpr int kBwTile = kBwGroups * kBlock;  // 8192 elements
constexpr int kBwStages = 2;
constexpr size_t kBwStageBytes = (size_t)kBwTile * (4 + 4 + 1 + 1);  // p, g, m_code, v_code

// The maps and midpoints are gathered at data-dependent indices; each is held
// kMapCopies times, a copy kCopyShift banks over from the previous, and lane
// l reads copy l % kMapCopies, which moves the bank conflicts of the gathers.
// Measured on GB300 (blockwise-1e9): two copies 16 banks apart 2.6 % faster
// than one, four copies 8 banks apart 2.3 %.
constexpr int kMapCopies = 2;
constexpr int kCopyShift = 16;
struct BlockwiseShared {
    float q1[kMapCopies][256 + kCopyShift], q2[kMapCopies][256 + kCopyShift];
    float mid1[kMapCopies][512 + kCopyShift], mid2[kMapCopies][512 + kCopyShift];  // +Inf padded
    uint8_t bucket1[kBuckets], bucket2[kBuckets];
    uint32_t warp_max[kBwGroups][2][2][8];  // [group][block parity][m, v][warp of the group]
    uint32_t red[2][32];
};
// What the consumers need to know about a work item, written by the producer
// into slot k % kBwSlots (k: the CTA's item count) before it signals the
// item's stage.  The consumers hand a stage back before they compute, so a
// slot must outlive its stage: the producer rewrites slot k % kBwSlots for
// item k + kBwSlots only after every consumer warp has handed back item
// k + kBwStages, which each does after finishing item k.
constexpr int kBwSlots = 2 * kBwStages;
struct BwItemInfo {
    BlockwiseArgs a;
    int64_t b0;    // first block of the item (a tile), or the short last block
    int32_t nblk;  // whole blocks in the tile; 0: the short last block
    int32_t codes; // the code arrays were staged
};
constexpr size_t kBwSmemBytes = kBwStages * kBwStageBytes + sizeof(BlockwiseShared) +
                                2 * kBwStages * sizeof(uint64_t) + kBwSlots * sizeof(BwItemInfo) +
                                sizeof(int64_t);

// Redo, with the IEEE divide, the codes of the values that need it.
__device__ __noinline__ uint2 requantise_fixup(float x0, float x1, float x2, float x3, float x4,
                                               float x5, float x6, float x7, float scale,
                                               uint32_t floor, const float *mid, uint2 code)
{
    const float x[8] = {x0, x1, x2, x3, x4, x5, x6, x7};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (needs_ieee_divide(x[j], floor)) {
            const uint32_t cj = (uint32_t)count_below(mid, __fdiv_rn(x[j], scale));
            const int sh = 8 * (j & 3);
            if (j < 4)
                code.x = (code.x & ~(0xFFu << sh)) | (cj << sh);
            else
                code.y = (code.y & ~(0xFFu << sh)) | (cj << sh);
        }
    return code;
}

// Codes of a thread's 8 values of one moment, block scale bits sb in the
// FMA-division range.  Values that may need the IEEE divide (|x| below the
// floor: tiny x, and zeros, whose fast code is right anyway) send the thread
// through a fix-up pass that is rarely entered; one compare per value.
template <int K>
__device__ __forceinline__ uint2 requantise_fast(const float *x, uint32_t sb, const float *mid,
                                                 const uint8_t *table, int k)
{
    const float scale = __uint_as_float(sb), y = reciprocal_rn(scale);
    const float2 y2 = make_float2(y, y), ns2 = make_float2(-scale, -scale);
    const uint32_t floor = fast_quotient_floor(sb);
    const float floorf = __uint_as_float(floor);
    uint2 code = make_uint2(0u, 0u);
    bool fix = false;
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        fix = fix || fabsf(x[j]) < floorf || fabsf(x[j + 1]) < floorf;
        const float2 c = divide_pair_for_code(make_float2(x[j], x[j + 1]), ns2, y2);
        const uint32_t cj = code_by_bucket<K>(mid, table, c.x, k) |
                            code_by_bucket<K>(mid, table, c.y, k) << 8;
        if (j < 4)
            code.x |= cj << (8 * j);
        else
            code.y |= cj << (8 * (j - 4));
    }
    if (fix)
        code = requantise_fixup(x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7], scale, floor, mid,
                                code);
    return code;
}

// One 2048-element block b, by one group of 256 threads (thread gt of the
// group holds elements 4gt..4gt+3 and 1024+4gt..1024+4gt+3: pv, gv, and the
// codes mc, vc packed four to a word; amv the block's two absmax values, read
// before the stage was handed back).  WHOLE: every element is in range (all
// blocks but a short last one), so no per-element bound logic is compiled in.
// The update is adamw_vector's (packed pairs of elements, one warp vote for
// the branch-free quotients per four), the requantiser's divisions packed in
// pairs too: 4 % faster on GB300 than one element at a time with the IEEE
// arithmetic.  (Pairing an element's two moments instead measured slower: the
// kernel is at its register limit.)  The block absmax is a warp max
// (redux.sync on the binary32 bits of |x|, which orders non-negative floats and
// lets a NaN win) and a max over the group's 8 warps through shared memory,
// between which the group meets at its named barrier; `gpar` alternates the
// shared slots between consecutive blocks of the group.
template <bool WHOLE, int K>
__device__ __forceinline__ void blockwise_block(const BlockwiseArgs &a, BlockwiseShared &sh,
                                                int64_t b, int group, int gt, uint32_t gpar,
                                                float2 amv, const float pv[8], const float gv[8],
                                                const uint32_t mc[2], const uint32_t vc[2],
                                                const Scalars &s, const ZeroSafe &zs, int k1,
                                                int k2, uint32_t &bad)
{
    const int lane = gt & 31, warp = gt >> 5, copy = lane % kMapCopies;
    const int64_t base = b * kBlock;
    float2 nv[8];  // (m', v') of the thread's 8 elements
    uint32_t um = 0, uv = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t e0 = base + 1024 * h + 4 * gt;
        float po[4], m[4], v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m[j] = __fmul_rn(sh.q1[copy][__byte_perm(mc[h], 0u, 0x4440u + j)], amv.x);
            v[j] = __fmul_rn(sh.q2[copy][__byte_perm(vc[h], 0u, 0x4440u + j)], amv.y);
        }
        Moments o[4];
        {
            const float2 P2[2] = {make_float2(pv[4 * h], pv[4 * h + 1]), make_float2(pv[4 * h + 2], pv[4 * h + 3])};
            const float2 G2[2] = {make_float2(gv[4 * h], gv[4 * h + 1]), make_float2(gv[4 * h + 2], gv[4 * h + 3])};
            const float2 M2[2] = {make_float2(m[0], m[1]), make_float2(m[2], m[3])};
            const float2 V2[2] = {make_float2(v[0], v[1]), make_float2(v[2], v[3])};
            Moments2 o2[2];
            float2 unused[2];
            adamw_vector<false, false, false>(P2, G2, M2, V2, s, pairs_of(s), zs, o2, unused);
            if (WHOLE)
                bad += nonfinite_count4(o2);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                o[2 * j] = Moments{o2[j].p.x, o2[j].m.x, o2[j].v.x};
                o[2 * j + 1] = Moments{o2[j].p.y, o2[j].m.y, o2[j].v.y};
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            po[j] = o[j].p;
            float2 x = make_float2(o[j].m, o[j].v);
            if (!WHOLE) {
                if (e0 + j < a.n)
                    bad += any_nonfinite(o[j]);
                else
                    x = make_float2(0.0f, 0.0f);  // |0| never raises the block max
            }
            nv[4 * h + j] = x;
            um = max(um, __float_as_uint(x.x) & 0x7FFFFFFFu);
            uv = max(uv, __float_as_uint(x.y) & 0x7FFFFFFFu);
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(po[0], po[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(po[2], po[3]);
        if (WHOLE) {
            uint2 packed;
            packed.x = *reinterpret_cast<const uint32_t *>(&lo);
            packed.y = *reinterpret_cast<const uint32_t *>(&hi);
            __stcs(reinterpret_cast<uint2 *>(a.p_bf16 + e0), packed);
        } else {
            const __nv_bfloat16 hv[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e0 + j < a.n)
                    a.p_bf16[e0 + j] = *reinterpret_cast<const uint16_t *>(&hv[j]);
        }
    }
    // block absmax of m' and v' (NaN bits win the unsigned max)
    um = __reduce_max_sync(0xFFFFFFFFu, um);
    uv = __reduce_max_sync(0xFFFFFFFFu, uv);
    if (lane == 0) {
        sh.warp_max[group][gpar][0][warp] = um;
        sh.warp_max[group][gpar][1][warp] = uv;
    }
    asm volatile("bar.sync %0, 256;" ::"r"(1 + group) : "memory");
    um = __reduce_max_sync(0xFFFFFFFFu, lane < 8 ? sh.warp_max[group][gpar][0][lane] : 0u);
    uv = __reduce_max_sync(0xFFFFFFFFu, lane < 8 ? sh.warp_max[group][gpar][1][lane] : 0u);
    if (gt == 0) {
        a.m_absmax[b] = __uint_as_float(um);
        a.v_absmax[b] = __uint_as_float(uv);
    }
    const uint32_t floor_bits = __float_as_uint(1e-30f);
    const uint32_t smb = max(um, floor_bits), svb = max(uv, floor_bits);  // NaN bits stay NaN
    float xm[8], xv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        xm[j] = nv[j].x;
        xv[j] = nv[j].y;
    }
    const uint2 cm = scale_in_fast_range(smb)  // uniform over the group
                         ? requantise_fast<K>(xm, smb, sh.mid1[copy], sh.bucket1, k1)
                         : requantise_slow(xm[0], xm[1], xm[2], xm[3], xm[4], xm[5], xm[6], xm[7],
                                           __uint_as_float(smb), sh.mid1[copy]);
    const uint2 cv = scale_in_fast_range(svb)
                         ? requantise_fast<K>(xv, svb, sh.mid2[copy], sh.bucket2, k2)
                         : requantise_slow(xv[0], xv[1], xv[2], xv[3], xv[4], xv[5], xv[6], xv[7],
                                           __uint_as_float(svb), sh.mid2[copy]);
    const uint32_t mcode[2] = {cm.x, cm.y}, vcode[2] = {cv.x, cv.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t e0 = base + 1024 * h + 4 * gt;
        if (WHOLE) {
            *reinterpret_cast<uint32_t *>(a.m_code + e0) = mcode[h];
            *reinterpret_cast<uint32_t *>(a.v_code + e0) = vcode[h];
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e0 + j < a.n) {
                    a.m_code[e0 + j] = (uint8_t)(mcode[h] >> (8 * j));
                    a.v_code[e0 + j] = (uint8_t)(vcode[h] >> (8 * j));
                }
        }
    }
}

// Per-CTA set-up: maps, midpoints (+Inf padded) and the two bucket tables;
// returns the largest bucket population of each map.  Every thread of the CTA
// takes part.
__device__ __forceinline__ void blockwise_setup(BlockwiseShared &sh, const float *__restrict__ qmap1,
                                                const float *__restrict__ qmap2, int &k1, int &k2)
{
    const int tid = threadIdx.x;
    if (tid < 256) {
        for (int c = 0; c < kMapCopies; ++c) {
            sh.q1[c][tid] = __ldg(qmap1 + tid);
            sh.q2[c][tid] = __ldg(qmap2 + tid);
        }
    }
    __syncthreads();
    if (tid < 256) {
        const float a = tid < 255 ? __fmul_rn(__fadd_rn(sh.q1[0][tid], sh.q1[0][tid + 1]), 0.5f) : INFINITY;
        const float b = tid < 255 ? __fmul_rn(__fadd_rn(sh.q2[0][tid], sh.q2[0][tid + 1]), 0.5f) : INFINITY;
        for (int c = 0; c < kMapCopies; ++c) {
            sh.mid1[c][tid] = a;
            sh.mid2[c][tid] = b;
            sh.mid1[c][256 + tid] = INFINITY;
            sh.mid2[c][256 + tid] = INFINITY;
        }
    }
    __syncthreads();
    k1 = build_buckets(sh.mid1[0], sh.bucket1, sh.red[0]);
    k2 = build_buckets(sh.mid2[0], sh.bucket2, sh.red[1]);
    __syncthreads();
}

// One tensor of a blockwise list; item0 = its first work item in the list.
// A tensor's work items are its tiles of kBwGroups whole blocks (the last
// tile may hold fewer) and, when n is not a multiple of 2048, one more item:
// the short last block.
struct BwDesc {
    BlockwiseArgs a;
    int64_t item0;
};

__host__ __device__ __forceinline__ int64_t bw_full_tiles(int64_t n)
{
    return (n / kBlock + kBwGroups - 1) / kBwGroups;
}

template <bool MULTI>
struct BwCursor {
    const BwDesc *table;
    int32_t ntensors, t;
    int64_t next;
    BwDesc d;
    __device__ __forceinline__ BwCursor(const BwDesc *tab, int32_t nt, int64_t total, const BwDesc &single)
        : table(tab), ntensors(nt), t(0), next(total), d(single)
    {
        if (MULTI) {
            d = table[0];
            next = ntensors > 1 ? table[1].item0 : total;
        }
    }
    __device__ __forceinline__ void seek(int64_t c, int64_t total)
    {
        if (MULTI)
            while (c >= next) {
                ++t;
                d = table[t];
                next = t + 1 < ntensors ? table[t + 1].item0 : total;
            }
    }
};

__device__ __forceinline__ bool codes_staged(const BlockwiseArgs &a)
{
    return ((reinterpret_cast<uintptr_t>(a.m_code) | reinterpret_cast<uintptr_t>(a.v_code)) & 15u) == 0;
}

// Stage an item: write its slot and issue its bulk copies into stage
// j % kBwStages (j: the CTA's item count).  Issued by thread 0 for the first
// two items and afterwards by the consumer warp whose release completes a
// stage, so the kernel needs no producer warp.
// `cur` is the shared table position: written by whichever thread issues,
// possibly out of order, but every value written is the tensor of an item at
// or before any later one, and the walk only moves forward from it.
template <bool MULTI>
__device__ __forceinline__ void bw_issue(unsigned char *smem, uint64_t *full, BwItemInfo *info,
                                         const BwDesc *table, int32_t ntensors,
                                         const BwDesc &single, volatile int32_t *cur, int64_t j)
{
    const int64_t c = blockIdx.x + j * (int64_t)gridDim.x;
    const int st = (int)(j % kBwStages);
    const BwDesc *dp = &single;
    if (MULTI) {
        int32_t t = *cur;
        while (t + 1 < ntensors && c >= table[t + 1].item0)
            ++t;
        *cur = t;
        dp = table + t;
    }
    const BlockwiseArgs a = dp->a;
    const int64_t kt = c - dp->item0;
    const int64_t nf = a.n / kBlock;
    BwItemInfo &it = info[j % kBwSlots];
    it.a = a;
    if (kt < bw_full_tiles(a.n)) {
        const int64_t b0 = kt * kBwGroups;
        const int64_t nb = nf - b0 < kBwGroups ? nf - b0 : kBwGroups;
        const uint32_t elems = (uint32_t)(nb * kBlock);
        const int64_t e0 = b0 * kBlock;
        const bool codes = codes_staged(a);
        it.b0 = b0;
        it.nblk = (int32_t)nb;
        it.codes = codes ? 1 : 0;
        mbar_arrive_expect(&full[st], elems * (codes ? 10u : 8u));  // releases the slot too
        unsigned char *buf = smem + (size_t)st * kBwStageBytes;
        bulk_load(buf, a.p + e0, elems * 4u, &full[st]);
        bulk_load(buf + kBwTile * 4, a.g + e0, elems * 4u, &full[st]);
        if (codes) {
            bulk_load(buf + kBwTile * 8, a.m_code + e0, elems, &full[st]);
            bulk_load(buf + kBwTile * 9, a.v_code + e0, elems, &full[st]);
        }
    } else {  // the short last block: read from global memory
        it.b0 = nf;
        it.nblk = 0;
        it.codes = 0;
        mbar_arrive_expect(&full[st], 0u);
    }
}

// One release of stage st by a warp (lane 0); true for the warp whose release
// completes it, which then owns the stage: every warp's reads of it are
// ordered before the release (acquire-release counter), and the proxy fence
// orders them before the bulk copies that will overwrite it.
__device__ __forceinline__ bool bw_release(uint32_t *count)
{
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "r"(smem_addr(count))
                 : "memory");
    if (old != (uint32_t)(kBwWarps - 1))
        return false;
    *count = 0u;  // no release of this stage's next use precedes its refill
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    return true;
}

template <bool MULTI>
__device__ __forceinline__ void bw_consume(unsigned char *smem, uint64_t *full, uint32_t *released,
                                           BlockwiseShared &sh, BwItemInfo *info,
                                           const BwDesc *table, int32_t ntensors,
                                           const BwDesc &single, volatile int32_t *cur,
                                           int64_t total, int64_t items, const Scalars &s, int k1,
                                           int k2, uint32_t &bad)
{
    const int group = threadIdx.x >> 8, gt = threadIdx.x & 255;
    const int kmax = k1 > k2 ? k1 : k2;
    const ZeroSafe zs = zero_safe_of(s);
    uint32_t gpar = 0;
    for (int64_t k = 0; k < items; ++k) {
        const int st = (int)(k % kBwStages);
        if (!mbar_wait(&full[st], (uint32_t)((k / kBwStages) & 1))) {
            pipe_fault(kFaultFullWait);
            break;
        }
        const BwItemInfo &it = info[k % kBwSlots];
        const BlockwiseArgs &a = it.a;  // read from the slot where used
        const bool tile = it.nblk > 0;
        const int64_t b = tile ? it.b0 + group : it.b0;
        const bool mine = tile ? group < it.nblk : group == 0;
        // the block's absmax values first (their loads overlap the copies below)
        float2 amv = make_float2(0.0f, 0.0f);
        if (mine)
            amv = make_float2(a.m_absmax[b], a.v_absmax[b]);
        // this thread's elements and codes, into registers
        float pv[8], gv[8];
        uint32_t mc[2] = {0u, 0u}, vc[2] = {0u, 0u};
        if (tile && mine) {
            const unsigned char *buf = smem + (size_t)st * kBwStageBytes;
            const int o = group * kBlock + 4 * gt;
            const bool codes = it.codes != 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 x = *reinterpret_cast<const float4 *>(buf + 4 * (o + 1024 * h));
                const float4 y = *reinterpret_cast<const float4 *>(buf + kBwTile * 4 + 4 * (o + 1024 * h));
                pv[4 * h] = x.x; pv[4 * h + 1] = x.y; pv[4 * h + 2] = x.z; pv[4 * h + 3] = x.w;
                gv[4 * h] = y.x; gv[4 * h + 1] = y.y; gv[4 * h + 2] = y.z; gv[4 * h + 3] = y.w;
                if (codes) {
                    mc[h] = *reinterpret_cast<const uint32_t *>(buf + kBwTile * 8 + o + 1024 * h);
                    vc[h] = *reinterpret_cast<const uint32_t *>(buf + kBwTile * 9 + o + 1024 * h);
                } else {
                    const int64_t e = b * kBlock + 1024 * h + 4 * gt;
                    mc[h] = *reinterpret_cast<const uint32_t *>(a.m_code + e);
                    vc[h] = *reinterpret_cast<const uint32_t *>(a.v_code + e);
                }
            }
        } else if (mine) {  // the short last block, from global memory
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t e0 = b * kBlock + 1024 * h + 4 * gt;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = e0 + j < a.n;
                    pv[4 * h + j] = in ? a.p[e0 + j] : 0.0f;
                    gv[4 * h + j] = in ? a.g[e0 + j] : 0.0f;
                    mc[h] |= (in ? (uint32_t)a.m_code[e0 + j] : 0u) << (8 * j);
                    vc[h] |= (in ? (uint32_t)a.v_code[e0 + j] : 0u) << (8 * j);
                }
            }
        }
        // the stage is no longer read: hand it back before computing; the last
        // warp to do so refills it with the item kBwStages ahead
        __syncwarp();
        if ((threadIdx.x & 31) == 0 && bw_release(&released[st]) && k + kBwStages < items)
            bw_issue<MULTI>(smem, full, info, table, ntensors, single, cur, k + kBwStages);
        if (mine) {
            // whole blocks with at most one midpoint per bucket (the log-linear
            // maps): the specialised body; anything else: the generic one
            if (tile && kmax <= 1)
                blockwise_block<true, 1>(a, sh, b, group, gt, gpar, amv, pv, gv, mc, vc, s, zs, k1,
                                         k2, bad);
            else
                blockwise_block<false, 0>(a, sh, b, group, gt, gpar, amv, pv, gv, mc, vc, s, zs, k1,
                                          k2, bad);
            gpar ^= 1u;
        }
    }
}

// The blockwise step over a tensor list (MULTI) or one tensor.  One CTA of 32
// warps per SM: four groups of 8 warps update one block each of a tile of
// kBwGroups blocks staged (p, g and, when both code arrays are 16-byte
// aligned, the two code arrays) by bulk copies into a two-stage ring; the
// warp whose release completes a stage issues the copies of its next item.
template <bool MULTI>
__global__ void __launch_bounds__(kBwThreads, 1)
blockwise8_pipe_kernel(const BwDesc *__restrict__ table, int32_t ntensors, int64_t total_items,
                       const BwDesc single, const float *__restrict__ qmap1,
                       const float *__restrict__ qmap2, const Scalars s,
                       unsigned long long *nonfinite)
{
    extern __shared__ __align__(128) unsigned char bw_smem[];
    BlockwiseShared &sh = *reinterpret_cast<BlockwiseShared *>(bw_smem + kBwStages * kBwStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(bw_smem + kBwStages * kBwStageBytes + sizeof(BlockwiseShared));
    uint32_t *released = reinterpret_cast<uint32_t *>(full + kBwStages);  // kBwStages counters
    BwItemInfo *info = reinterpret_cast<BwItemInfo *>(full + 2 * kBwStages);
    volatile int32_t *cur = reinterpret_cast<volatile int32_t *>(info + kBwSlots);
    // this CTA's items: blockIdx.x, blockIdx.x + gridDim.x, ...
    const int64_t items = total_items > blockIdx.x
                              ? (total_items - blockIdx.x + gridDim.x - 1) / gridDim.x
                              : 0;
    int k1, k2;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kBwStages; ++i) {
            mbar_init(&full[i], 1);
            released[i] = 0u;
        }
        *cur = 0;
        mbar_init_fence();
    }
    blockwise_setup(sh, qmap1, qmap2, k1, k2);  // ends with __syncthreads
    if (threadIdx.x == 0)
        for (int64_t j = 0; j < kBwStages && j < items; ++j)
            bw_issue<MULTI>(bw_smem, full, info, table, ntensors, single, cur, j);
    uint32_t bad = 0;
    bw_consume<MULTI>(bw_smem, full, released, sh, info, table, ntensors, single, cur,
                      total_items, items, s, k1, k2, bad);
    flush_nonfinite(bad, nonfinite);
}

}  // namespace pa

#include "turbo.cuh"

// ===========================================================================
// Host side
// ===========================================================================
namespace {

using pa::Desc;
using pa::Scalars;

thread_local std::string g_last_error;

pa_status fail(pa_status code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

pa_status ok()
{
    g_last_error.clear();
    return PA_OK;
}

pa_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Hyperparameters -> FP32 scalars: each formed in double, rounded once to
// float (KBench quantized_adamw_step forms them in double precision).
// step is the 1-based global step ("Execution contract": one global step).
pa_status make_scalars(int64_t step, double lr, double beta1, double beta2, double eps,
                       double wd, Scalars *s)
{
    if (step < 1)
        return fail(PA_ERR_ARG, "step must be >= 1 (got %lld)", (long long)step);
    if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(wd) ||
        !std::isfinite(beta1) || !std::isfinite(beta2))
        return fail(PA_ERR_ARG, "hyperparameters must be finite");
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
        return fail(PA_ERR_ARG, "betas must lie in [0, 1) (got %g, %g)", beta1, beta2);
    if (eps < 0.0)
        return fail(PA_ERR_ARG, "eps must be >= 0 (got %g)", eps);
    s->b1 = (float)beta1;
    s->b2 = (float)beta2;
    s->c1 = (float)(1.0 - beta1);
    s->c2 = (float)(1.0 - beta2);
    s->bc2 = (float)(1.0 - std::pow(beta2, (double)step));
    s->ss = (float)(lr / (1.0 - std::pow(beta1, (double)step)));
    s->dk = (float)(1.0 - lr * wd);
    s->ef = (float)eps;
    return PA_OK;
}

// ---- per-device launch geometry --------------------------------------------
// Kernels launched with kThreads threads and no dynamic shared memory: the
// register-staged step (on host memory) and the codecs.
enum KernelSlot { kSlotHostE4, kSlotCodec, kSlotTurbo, kNumSlots };

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int occ[kNumSlots] = {0};  // resident CTAs per SM, by kernel slot
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

const void *kernel_of(int slot)
{
    switch (slot) {
    case kSlotHostE4: return (const void *)pa::adamw_step_kernel<pa::kE4, false, false, float>;
    case kSlotTurbo: return (const void *)pa::turbo_step_kernel;
    default: return (const void *)pa::encode_state_kernel<pa::kE4>;
    }
}

// Persistent grid size for a kernel on the current device: resident CTAs per
// SM times the SM count, capped by the work items.
pa_status grid_for(int slot, int64_t work, int *grid)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.ready) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        for (int k = 0; k < kNumSlots; ++k) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.occ[k], kernel_of(k), pa::kThreads, 0);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            if (di.occ[k] < 1)
                di.occ[k] = 1;
        }
        di.ready = true;
    }
    const int64_t full = (int64_t)di.sms * di.occ[slot];
    *grid = (int)(work < full ? (work > 0 ? work : 1) : full);
    return PA_OK;
}

// Elements per chunk for a launch over `elements` parameters: as many waves
// (at most kMaxWaves) as keep at least 32 chunks per resident CTA, so that
// large launches amortise the per-chunk set-up and small ones still spread
// over every SM.
pa_status chunk_size(int slot, int64_t elements, int64_t *chunk)
{
    int full = 0;
    pa_status st = grid_for(slot, INT64_MAX, &full);
    if (st != PA_OK)
        return st;
    int64_t waves = elements / (pa::kWave * (int64_t)full * 32);
    waves = waves < 1 ? 1 : (waves > pa::kMaxWaves ? pa::kMaxWaves : waves);
    *chunk = waves * pa::kWave;
    return PA_OK;
}

// Grid of a staged kernel: one CTA per SM (its shared-memory ring takes most
// of the SM), capped by the tiles.  The first launch of each kernel on a device
// raises its dynamic shared-memory limit to `smem`, the most any launch of it
// uses (a launch passes what it needs: the descriptor copy depends on the list).
pa_status pipe_grid(const void *kernel, size_t smem, int64_t tiles, int *grid,
                    int threads = pa::kPipeThreads)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "device ordinal %d out of range", dev);
    static std::mutex mu;
    static std::vector<std::pair<const void *, int>> ready;  // (kernel, device) set up
    static int sms[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    bool done = false;
    for (const auto &r : ready)
        done = done || (r.first == kernel && r.second == dev);
    if (!done) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "raising the shared-memory limit of the staged step");
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (occ < 1)
            return fail(PA_ERR_CUDA, "the staged step (%zu bytes of shared memory) does not fit an SM",
                        smem);
        if (sms[dev] == 0 &&
            (e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        ready.emplace_back(kernel, dev);
    }
    const int64_t full = sms[dev];
    *grid = (int)(tiles < full ? (tiles > 0 ? tiles : 1) : full);
    return PA_OK;
}

// Elements per tile of a staged launch over `elements` parameters in `tiles`
// tiles of kTile: kTile, unless those tiles would leave SMs idle; then the
// smallest multiple of 256 (at least 256) that spreads the elements over the
// SMs, so a small workload runs on many SMs at once instead of one.
pa_status launch_tile(int64_t tiles, int64_t elements, int32_t *tile)
{
    *tile = pa::kTile;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (tiles >= sms || sms < 1)
        return PA_OK;
    int64_t t = (elements + sms - 1) / sms;
    t = (t + 255) / 256 * 256;
    *tile = (int32_t)(t < 256 ? 256 : (t > pa::kTile ? pa::kTile : t));
    return PA_OK;
}

// Launch the staged step over `tiles` tiles (table == nullptr: the one tensor
// `single`).  A launch of fewer than kPairedTileRounds tiles per CTA takes the
// instantiation whose whole tiles also run the branch-free arithmetic in
// packed pairs (PAIR 2): measured on GB300, the 9.7M-parameter gpt-52 list
// 4 % faster that way, a 2^28-parameter flat tensor 4 % slower (HBM-bound,
// its whole tiles keep the scalar arm).  Bfloat16 gradients always pair.
constexpr int64_t kPairedTileRounds = 32;

template <int MODE, typename GT, bool U1, int PAIR>
void launch_pipe_as(int grid, size_t used, const Desc *table, int32_t ntensors, int64_t tiles,
                    const Desc &single, const Scalars &s, unsigned long long *nonfinite,
                    int32_t tile, pa_stream stream)
{
    pa::adamw_step_pipe_kernel<MODE, U1, GT, PAIR><<<grid, pa::kPipeThreads, used, (cudaStream_t)stream>>>(
        table, ntensors, tiles, single, s, nonfinite, tile);
}

template <int MODE, typename GT>
pa_status launch_pipe(const Desc *table, int32_t ntensors, int64_t tiles, const Desc &single,
                      const Scalars &s, unsigned long long *nonfinite, int32_t tile, size_t used,
                      pa_stream stream)
{
    const size_t smem = pa::PipeLayout<MODE, GT>::kBytes;  // the kernel's limit
    const bool u1 = s.bc2 == 1.0f;
    int grid = 0;
    pa_status st = pipe_grid(u1 ? (const void *)pa::adamw_step_pipe_kernel<MODE, true, GT>
                                : (const void *)pa::adamw_step_pipe_kernel<MODE, false, GT>,
                             smem, tiles, &grid);
    if (st != PA_OK)
        return st;
    if constexpr (sizeof(GT) == 4) {
        if (tiles < kPairedTileRounds * (int64_t)grid) {
            // same shared memory and block; its own attribute and occupancy check
            int g2 = 0;
            st = pipe_grid(u1 ? (const void *)pa::adamw_step_pipe_kernel<MODE, true, GT, 2>
                              : (const void *)pa::adamw_step_pipe_kernel<MODE, false, GT, 2>,
                           smem, tiles, &g2);
            if (st != PA_OK)
                return st;
            grid = g2 < grid ? g2 : grid;
            if (u1)
                launch_pipe_as<MODE, GT, true, 2>(grid, used, table, ntensors, tiles, single, s,
                                                  nonfinite, tile, stream);
            else
                launch_pipe_as<MODE, GT, false, 2>(grid, used, table, ntensors, tiles, single, s,
                                                   nonfinite, tile, stream);
            return PA_OK;
        }
    }
    if (u1) {
        launch_pipe_as<MODE, GT, true, 1>(grid, used, table, ntensors, tiles, single, s, nonfinite, tile, stream);
    } else {
        launch_pipe_as<MODE, GT, false, 1>(grid, used, table, ntensors, tiles, single, s, nonfinite, tile, stream);
    }
    return PA_OK;
}

pa_status check_launch(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, what);
    return ok();
}

// ---- descriptors -------------------------------------------------------------
// Fill d for one tensor; returns its chunk count.  The 16-byte path needs p, g
// and the state (and v in FP32 mode) to share their address modulo 16; the
// head peels the elements before the first 16-byte boundary.
int64_t describe(const pa_tensor &t, int mode, int64_t chunk, Desc *d, int grad_bytes = 4)
{
    d->p = t.p;
    d->g = t.g;
    d->s1 = t.state;
    d->s2 = t.state2;
    d->n = t.n;
    // element phase within a 4-element vector: all streams must agree for the
    // vector path (p and the state are 4-byte elements, g 4 or 2 bytes)
    const uintptr_t ph = (reinterpret_cast<uintptr_t>(t.p) >> 2) & 3u;
    const uintptr_t gph = (reinterpret_cast<uintptr_t>(t.g) / (uintptr_t)grad_bytes) & 3u;
    bool same = gph == ph && (reinterpret_cast<uintptr_t>(t.p) & 3u) == 0 &&
                (reinterpret_cast<uintptr_t>(t.p) & 15u) == 4 * ph &&
                (reinterpret_cast<uintptr_t>(t.g) & (uintptr_t)(4 * grad_bytes - 1)) ==
                    (uintptr_t)grad_bytes * gph &&
                (reinterpret_cast<uintptr_t>(t.state) & 15u) == 4 * ph;
    if (mode == pa::kF32)
        same = same && (reinterpret_cast<uintptr_t>(t.state2) & 15u) == 4 * ph;
    int64_t head = same ? (int64_t)((4u - ph) & 3u) : 0;
    // the staged body starts 16-byte aligned in every stream (a bfloat16
    // gradient can share p's element phase and still be 8 bytes off)
    same = same && ((reinterpret_cast<uintptr_t>(t.g) + (uintptr_t)grad_bytes * (uintptr_t)head) & 15u) == 0;
    if (!same)
        head = 0;
    d->vec = same ? 1 : 0;
    if (head > t.n)
        head = t.n;
    d->head = (int32_t)head;
    if (t.n == 0)
        return 0;
    const int64_t body = same ? t.n - head : t.n;
    const int64_t chunks = (body + chunk - 1) / chunk;
    return chunks > 0 ? chunks : 1;
}

pa_status check_tensor(const pa_tensor &t, int mode, int index, uintptr_t grad_align = 4)
{
    if (t.n < 0)
        return fail(PA_ERR_ARG, "tensor %d: n must be >= 0 (got %lld)", index, (long long)t.n);
    if (t.n == 0)
        return PA_OK;
    if (!t.p || !t.g || !t.state || (mode == pa::kF32 && !t.state2))
        return fail(PA_ERR_NULL, "tensor %d: NULL pointer with n = %lld", index, (long long)t.n);
    if (!aligned(t.p, 4) || !aligned(t.g, grad_align) || !aligned(t.state, 4) ||
        (mode == pa::kF32 && !aligned(t.state2, 4)))
        return fail(PA_ERR_ALIGN, "tensor %d: pointers must be aligned to their element size",
                    index);
    return PA_OK;
}

pa_status check_counter(const unsigned long long *nonfinite)
{
    if (nonfinite && !aligned(nonfinite, 8))
        return fail(PA_ERR_ALIGN, "nonfinite counter must be 8-byte aligned");
    return PA_OK;
}

template <int MODE, typename GT = float>
pa_status step_single(const pa_tensor &t, int64_t step, double lr, double beta1, double beta2,
                      double eps, double wd, unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if ((st = check_tensor(t, MODE, 0, sizeof(GT))) != PA_OK ||
        (st = check_counter(nonfinite)) != PA_OK)
        return st;
    if (t.n == 0)
        return ok();
    Desc d;
    int64_t tiles = describe(t, MODE, pa::kTile, &d, (int)sizeof(GT));
    int32_t tile = pa::kTile;
    if ((st = launch_tile(tiles, t.n, &tile)) != PA_OK)
        return st;
    if (tile != pa::kTile)
        tiles = describe(t, MODE, tile, &d, (int)sizeof(GT));
    d.chunk0 = 0;
    const size_t used = pa::PipeLayout<MODE, GT>::bytes_for(1);  // the descriptor, by value
    if ((st = launch_pipe<MODE, GT>(nullptr, 1, tiles, d, s, nonfinite, tile, used, stream)) != PA_OK)
        return st;
    return check_launch("adamw_step_pipe_kernel launch");
}

// ---- cached device descriptor tables (multi-tensor calls) -----------------------
// A list is uploaded once per device and reused while it is unchanged, so a
// training loop that steps the same tensors pays no host-to-device copy.  The
// table of a list is immutable once uploaded, so calls on different streams
// never see a table change under them.  A table that the graph-replayable step
// has used is pinned: a captured launch holds its address, so the
// least-recently-used eviction never frees it (only pa_release_tables does).
struct Table {
    int device;
    int mode;
    int grad_bytes;
    int64_t chunk;
    std::vector<Desc> host;
    Desc *dev;
    int64_t chunks;
    uint64_t last_use;
    bool pinned;
};

std::mutex g_tab_mu;
std::vector<Table> g_tables;
uint64_t g_tick = 0;
constexpr size_t kMaxTables = 64;

pa_status table_for(const pa_tensor *list, int32_t ntensors, int mode, int64_t chunk,
                    const Desc **dev_table, int64_t *chunks, int grad_bytes = 4,
                    bool pin = false)
{
    std::vector<Desc> host((size_t)ntensors);
    int64_t total = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        const int64_t c = describe(list[i], mode, chunk, &host[(size_t)i], grad_bytes);
        host[(size_t)i].chunk0 = total;
        total += c;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_tab_mu);
    ++g_tick;
    for (Table &t : g_tables) {
        if (t.device == dev && t.mode == mode && t.grad_bytes == grad_bytes && t.chunk == chunk &&
            t.host.size() == host.size() &&
            std::memcmp(t.host.data(), host.data(), host.size() * sizeof(Desc)) == 0) {
            t.last_use = g_tick;
            t.pinned = t.pinned || pin;
            *dev_table = t.dev;
            *chunks = t.chunks;
            return PA_OK;
        }
    }
    if (g_tables.size() >= kMaxTables) {  // free the least recently used unpinned list
        size_t old = g_tables.size();
        for (size_t k = 0; k < g_tables.size(); ++k)
            if (!g_tables[k].pinned &&
                (old == g_tables.size() || g_tables[k].last_use < g_tables[old].last_use))
                old = k;
        if (old < g_tables.size()) {
            int cur = dev;
            cudaSetDevice(g_tables[old].device);
            cudaFree(g_tables[old].dev);  // synchronises that device: no kernel still reads it
            cudaSetDevice(cur);
            g_tables.erase(g_tables.begin() + (long)old);
        }
    }
    Table t;
    t.device = dev;
    t.mode = mode;
    t.grad_bytes = grad_bytes;
    t.chunk = chunk;
    t.chunks = total;
    t.last_use = g_tick;
    t.pinned = pin;
    t.dev = nullptr;
    const size_t bytes = host.size() * sizeof(Desc);
    e = cudaMalloc((void **)&t.dev, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PA_ERR_NOMEM, "cudaMalloc of a %zu-byte descriptor table: %s", bytes,
                    cudaGetErrorString(e));
    }
    // synchronous copy: the table is complete before any kernel can read it
    e = cudaMemcpy(t.dev, host.data(), bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(t.dev);
        return cuda_fail(e, "descriptor table upload");
    }
    t.host = std::move(host);
    g_tables.push_back(std::move(t));
    *dev_table = g_tables.back().dev;
    *chunks = g_tables.back().chunks;
    return PA_OK;
}

template <int MODE, typename GT = float>
pa_status step_multi(const pa_tensor *list, int32_t ntensors, int64_t step, double lr,
                     double beta1, double beta2, double eps, double wd,
                     unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (ntensors < 0)
        return fail(PA_ERR_ARG, "ntensors must be >= 0 (got %d)", ntensors);
    if (ntensors == 0)
        return ok();
    if (!list)
        return fail(PA_ERR_NULL, "tensor list is NULL with ntensors = %d", ntensors);
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    int64_t total = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        if ((st = check_tensor(list[i], MODE, i, sizeof(GT))) != PA_OK)
            return st;
        total += list[i].n;
    }
    if (total == 0)
        return ok();
    // A one-tensor list goes by value in the launch's parameters: no table to
    // look up, allocate or upload, so a list whose pointers change from step
    // to step never meets cudaMalloc's or cudaMemcpy's synchronisation.
    if (ntensors == 1)
        return step_single<MODE, GT>(list[0], step, lr, beta1, beta2, eps, wd, nonfinite, stream);
    const Desc *table = nullptr;
    Desc none;
    std::memset(&none, 0, sizeof none);
    int64_t tiles = 0;
    for (int32_t i = 0; i < ntensors; ++i)
        tiles += (list[i].n + pa::kTile - 1) / pa::kTile;
    int32_t tile = pa::kTile;
    if ((st = launch_tile(tiles, total, &tile)) != PA_OK)
        return st;
    if ((st = table_for(list, ntensors, MODE, tile, &table, &tiles, (int)sizeof(GT))) != PA_OK)
        return st;
    const size_t used = pa::PipeLayout<MODE, GT>::bytes_for(ntensors);
    if ((st = launch_pipe<MODE, GT>(table, ntensors, tiles, none, s, nonfinite, tile, used, stream)) !=
        PA_OK)
        return st;
    return check_launch("adamw_step_pipe_kernel (multi) launch");
}

// True when m, rms and the words share their address modulo 16 (4-byte
// aligned each): the vectorised codec kernels then apply, after `head` < 4
// leading elements.
bool vector_codec(const void *m, const void *rms, const void *word, int64_t n, int64_t *head)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(m) & 15u;
    if ((reinterpret_cast<uintptr_t>(rms) & 15u) != a || (reinterpret_cast<uintptr_t>(word) & 15u) != a)
        return false;
    const int64_t h = (int64_t)((16u - a) & 15u) / 4;
    if (n < h + 4)
        return false;
    *head = h;
    return true;
}

template <int MODE>
pa_status encode(const float *m, const float *rms, uint32_t *word, int64_t n,
                 unsigned long long *nonfinite, pa_stream stream)
{
    if (n < 0)
        return fail(PA_ERR_ARG, "n must be >= 0 (got %lld)", (long long)n);
    if (n == 0)
        return ok();
    if (!m || !rms || !word)
        return fail(PA_ERR_NULL, "NULL pointer with n = %lld", (long long)n);
    if (!aligned(m, 4) || !aligned(rms, 4) || !aligned(word, 4))
        return fail(PA_ERR_ALIGN, "pointers must be 4-byte aligned");
    pa_status st = check_counter(nonfinite);
    if (st != PA_OK)
        return st;
    int grid = 0;
    int64_t head = 0;
    if (vector_codec(m, rms, word, n, &head)) {
        const int64_t waves = ((n - head) / 4 + pa::kThreads * pa::kUnroll - 1) /
                              (pa::kThreads * pa::kUnroll);
        if ((st = grid_for(kSlotCodec, waves, &grid)) != PA_OK)
            return st;
        pa::encode_state_vec_kernel<MODE><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(
            m, rms, word, n, head, nonfinite);
        return check_launch("encode_state_vec_kernel launch");
    }
    if ((st = grid_for(kSlotCodec, (n + pa::kThreads - 1) / pa::kThreads, &grid)) != PA_OK)
        return st;
    pa::encode_state_kernel<MODE><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(m, rms, word, n, nonfinite);
    return check_launch("encode_state_kernel launch");
}

template <int MODE>
pa_status decode(const uint32_t *word, float *m, float *rms, int64_t n, pa_stream stream)
{
    if (n < 0)
        return fail(PA_ERR_ARG, "n must be >= 0 (got %lld)", (long long)n);
    if (n == 0)
        return ok();
    if (!m || !rms || !word)
        return fail(PA_ERR_NULL, "NULL pointer with n = %lld", (long long)n);
    if (!aligned(m, 4) || !aligned(rms, 4) || !aligned(word, 4))
        return fail(PA_ERR_ALIGN, "pointers must be 4-byte aligned");
    int grid = 0;
    pa_status st;
    int64_t head = 0;
    if (vector_codec(m, rms, word, n, &head)) {
        const int64_t waves = ((n - head) / 4 + pa::kThreads * pa::kUnroll - 1) /
                              (pa::kThreads * pa::kUnroll);
        if ((st = grid_for(kSlotCodec, waves, &grid)) != PA_OK)
            return st;
        pa::decode_state_vec_kernel<MODE><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(
            word, m, rms, n, head);
        return check_launch("decode_state_vec_kernel launch");
    }
    if ((st = grid_for(kSlotCodec, (n + pa::kThreads - 1) / pa::kThreads, &grid)) != PA_OK)
        return st;
    pa::decode_state_kernel<MODE><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(word, m, rms, n);
    return check_launch("decode_state_kernel launch");
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

int32_t pa_version(void) { return 10000; }

const char *pa_status_string(pa_status status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL";
    case PA_ERR_ARG: return "PA_ERR_ARG";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_NOMEM: return "PA_ERR_NOMEM";
    default: return "PA_ERR_UNKNOWN";
    }
}

const char *pa_last_error(void) { return g_last_error.c_str(); }

pa_status pa_encode_state(const float *m, const float *rms, uint32_t *word, int64_t n,
                          unsigned long long *nonfinite, pa_stream stream)
{
    return encode<pa::kE4>(m, rms, word, n, nonfinite, stream);
}

pa_status pa_decode_state(const uint32_t *word, float *m, float *rms, int64_t n, pa_stream stream)
{
    return decode<pa::kE4>(word, m, rms, n, stream);
}

pa_status pa_encode_state_fp16(const float *m, const float *rms, uint32_t *word, int64_t n,
                               unsigned long long *nonfinite, pa_stream stream)
{
    return encode<pa::kFP16>(m, rms, word, n, nonfinite, stream);
}

pa_status pa_decode_state_fp16(const uint32_t *word, float *m, float *rms, int64_t n,
                               pa_stream stream)
{
    return decode<pa::kFP16>(word, m, rms, n, stream);
}

pa_status pa_adamw_step_packed_e4(float *p, const float *g, uint32_t *state, int64_t n,
                                  int64_t step, double lr, double beta1, double beta2,
                                  double eps, double wd, unsigned long long *nonfinite,
                                  pa_stream stream)
{
    const pa_tensor t = {p, g, state, nullptr, n};
    return step_single<pa::kE4>(t, step, lr, beta1, beta2, eps, wd, nonfinite, stream);
}

pa_status pa_adamw_step_packed_fp16(float *p, const float *g, uint32_t *state, int64_t n,
                                    int64_t step, double lr, double beta1, double beta2,
                                    double eps, double wd, unsigned long long *nonfinite,
                                    pa_stream stream)
{
    const pa_tensor t = {p, g, state, nullptr, n};
    return step_single<pa::kFP16>(t, step, lr, beta1, beta2, eps, wd, nonfinite, stream);
}

pa_status pa_adamw_step_fp32(float *p, const float *g, float *m, float *v, int64_t n,
                             int64_t step, double lr, double beta1, double beta2, double eps,
                             double wd, unsigned long long *nonfinite, pa_stream stream)
{
    const pa_tensor t = {p, g, m, v, n};
    return step_single<pa::kF32>(t, step, lr, beta1, beta2, eps, wd, nonfinite, stream);
}

pa_status pa_adamw_step_packed_e4_multi(const pa_tensor *list, int32_t ntensors, int64_t step,
                                        double lr, double beta1, double beta2, double eps,
                                        double wd, unsigned long long *nonfinite,
                                        pa_stream stream)
{
    return step_multi<pa::kE4>(list, ntensors, step, lr, beta1, beta2, eps, wd, nonfinite, stream);
}

pa_status pa_adamw_step_packed_fp16_multi(const pa_tensor *list, int32_t ntensors,
                                          int64_t step, double lr, double beta1, double beta2,
                                          double eps, double wd, unsigned long long *nonfinite,
                                          pa_stream stream)
{
    return step_multi<pa::kFP16>(list, ntensors, step, lr, beta1, beta2, eps, wd, nonfinite,
                                 stream);
}

pa_status pa_adamw_step_fp32_multi(const pa_tensor *list, int32_t ntensors, int64_t step,
                                   double lr, double beta1, double beta2, double eps,
                                   double wd, unsigned long long *nonfinite, pa_stream stream)
{
    return step_multi<pa::kF32>(list, ntensors, step, lr, beta1, beta2, eps, wd, nonfinite, stream);
}

pa_status pa_adamw_step_blockwise8(const float *p, const float *g, uint16_t *p_bf16,
                                   uint8_t *m_code, float *m_absmax, uint8_t *v_code,
                                   float *v_absmax, const float *qmap1, const float *qmap2,
                                   int64_t n, int64_t step, double lr, double beta1,
                                   double beta2, double eps, double wd,
                                   unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (n < 0)
        return fail(PA_ERR_ARG, "n must be >= 0 (got %lld)", (long long)n);
    if (n == 0)
        return ok();
    if (!p || !g || !p_bf16 || !m_code || !m_absmax || !v_code || !v_absmax || !qmap1 || !qmap2)
        return fail(PA_ERR_NULL, "NULL pointer with n = %lld", (long long)n);
    if (!aligned(p, 16) || !aligned(g, 16))
        return fail(PA_ERR_ALIGN, "p and g must be 16-byte aligned");
    if (!aligned(p_bf16, 8))
        return fail(PA_ERR_ALIGN, "p_bf16 must be 8-byte aligned");
    if (!aligned(m_code, 4) || !aligned(v_code, 4))
        return fail(PA_ERR_ALIGN, "m_code and v_code must be 4-byte aligned");
    if (!aligned(m_absmax, 4) || !aligned(v_absmax, 4) || !aligned(qmap1, 4) || !aligned(qmap2, 4))
        return fail(PA_ERR_ALIGN, "absmax arrays and maps must be 4-byte aligned");
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    pa::BwDesc d;
    d.a = {p, g, p_bf16, m_code, m_absmax, v_code, v_absmax, n};
    d.item0 = 0;
    const int64_t items = pa::bw_full_tiles(n) + (n % pa::kBlock != 0 ? 1 : 0);
    int grid = 0;
    if ((st = pipe_grid((const void *)pa::blockwise8_pipe_kernel<false>, pa::kBwSmemBytes, items,
                        &grid, pa::kBwThreads)) != PA_OK)
        return st;
    pa::blockwise8_pipe_kernel<false><<<grid, pa::kBwThreads, pa::kBwSmemBytes, (cudaStream_t)stream>>>(
        nullptr, 1, items, d, qmap1, qmap2, s, nonfinite);
    return check_launch("blockwise8_pipe_kernel launch");
}

pa_status pa_shutdown(void)
{
    // the cached descriptor tables; the host-step streams and events live until exit
    return pa_release_tables();
}

pa_status pa_device_fault(uint32_t *code, int32_t clear)
{
    if (!code)
        return fail(PA_ERR_NULL, "code is NULL");
    cudaError_t e = cudaMemcpyFromSymbol(code, pa::g_pipe_fault, sizeof(uint32_t));
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the device fault flag");
    if (clear && *code != 0) {
        const uint32_t zero = 0;
        if ((e = cudaMemcpyToSymbol(pa::g_pipe_fault, &zero, sizeof zero)) != cudaSuccess)
            return cuda_fail(e, "clearing the device fault flag");
    }
    return ok();
}

pa_status release_blockwise_tables();

pa_status pa_release_tables(void)
{
    release_blockwise_tables();
    std::lock_guard<std::mutex> lock(g_tab_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (Table &t : g_tables) {
        cudaSetDevice(t.device);
        cudaFree(t.dev);
    }
    g_tables.clear();
    cudaSetDevice(cur);
    return ok();
}

}  // extern "C"

// ===========================================================================
// Multi-tensor packed-E4 step that allocates nothing
// ===========================================================================
// pa_adamw_step_packed_e4_multi keeps each list's descriptor table in device
// memory that the library obtains with cudaMalloc.  Some callers cannot let a
// library do that: a framework whose caching allocator has reserved the
// device's memory and expects every allocation to go through it, or a loop
// that must not meet cudaMalloc's and cudaFree's implicit synchronisation.
// For them this variant keeps the table in a fixed device array that is part
// of the library image: every device that loads the library holds the
// PA_NOALLOC_MAX_TENSORS descriptors (56 bytes each) until the process exits.
namespace {

constexpr int32_t kNoAllocMaxTensors = PA_NOALLOC_MAX_TENSORS;

}  // namespace

static __device__ __align__(256) pa::Desc g_noalloc_table[PA_NOALLOC_MAX_TENSORS];

// The descriptors reach the array as kernel parameters, up to kNoAllocBatch per
// launch (8 + 512 * 56 = 28,680 bytes, under the 32,764-byte parameter limit),
// written by a small kernel on the caller's stream: the launch copies its
// parameters when it is issued, so the host buffer is free again at once and
// nothing waits for the stream (a copy from pageable host memory would).
constexpr int kNoAllocBatch = 512;
struct NoAllocBatch {
    int32_t first;  // index of d[0] in the array
    int32_t count;  // descriptors in d
    pa::Desc d[kNoAllocBatch];
};

__global__ void noalloc_upload_kernel(const __grid_constant__ NoAllocBatch b)
{
    constexpr int kWords = sizeof(pa::Desc) / sizeof(uint64_t);
    const uint64_t *src = reinterpret_cast<const uint64_t *>(b.d);
    uint64_t *dst = reinterpret_cast<uint64_t *>(g_noalloc_table + b.first);
    for (int i = threadIdx.x; i < b.count * kWords; i += blockDim.x)
        dst[i] = src[i];
}

namespace {

std::mutex g_noalloc_mu;
pa::Desc *g_noalloc_ptr[64] = {nullptr};  // device address of the array, per device
thread_local NoAllocBatch g_noalloc_batch;

// The array's name is only a host-side stand-in in host code; its device
// address is looked up once per device, with that device current.
pa_status noalloc_table_address(pa::Desc **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_table);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress of the descriptor array");
        g_noalloc_ptr[dev] = static_cast<pa::Desc *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_adamw_step_packed_e4_multi_noalloc(
    const pa_tensor *list, int32_t ntensors, int64_t step, double lr, double beta1,
    double beta2, double eps, double wd, unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (ntensors < 0)
        return fail(PA_ERR_ARG, "ntensors must be >= 0 (got %d)", ntensors);
    if (ntensors > kNoAllocMaxTensors)
        return fail(PA_ERR_ARG,
                    "ntensors = %d exceeds the %d descriptors of the fixed device array; "
                    "use pa_adamw_step_packed_e4_multi or split the list",
                    ntensors, kNoAllocMaxTensors);
    if (ntensors == 0)
        return ok();
    if (!list)
        return fail(PA_ERR_NULL, "tensor list is NULL with ntensors = %d", ntensors);
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    int64_t total = 0, tiles = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        if ((st = check_tensor(list[i], pa::kE4, i)) != PA_OK)
            return st;
        total += list[i].n;
    }
    if (total == 0)
        return ok();
    pa::Desc *table = nullptr;
    if ((st = noalloc_table_address(&table)) != PA_OK)
        return st;
    // The whole used prefix is rewritten, in batches of kNoAllocBatch, so
    // nothing of an earlier call is read.
    NoAllocBatch &b = g_noalloc_batch;
    for (int32_t first = 0; first < ntensors; first += kNoAllocBatch) {
        b.first = first;
        b.count = ntensors - first < kNoAllocBatch ? ntensors - first : kNoAllocBatch;
        for (int32_t k = 0; k < b.count; ++k) {
            const int64_t c = describe(list[first + k], pa::kE4, pa::kTile, &b.d[k]);
            b.d[k].chunk0 = tiles;
            tiles += c;
        }
        noalloc_upload_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(b);
        if ((st = check_launch("descriptor upload to the fixed device array")) != PA_OK)
            return st;
    }
    const size_t smem = pa::PipeLayout<pa::kE4>::kBytes;  // the kernel's limit
    const size_t used = pa::PipeLayout<pa::kE4>::bytes_for(ntensors);
    const void *kern = s.bc2 == 1.0f ? (const void *)pa::adamw_step_pipe_kernel<pa::kE4, true>
                                     : (const void *)pa::adamw_step_pipe_kernel<pa::kE4, false>;
    int grid = 0;
    if ((st = pipe_grid(kern, smem, tiles, &grid)) != PA_OK)
        return st;
    pa::Desc none;
    std::memset(&none, 0, sizeof none);
    if (s.bc2 == 1.0f)
        pa::adamw_step_pipe_kernel<pa::kE4, true><<<grid, pa::kPipeThreads, used, (cudaStream_t)stream>>>(
            table, ntensors, tiles, none, s, nonfinite, pa::kTile);
    else
        pa::adamw_step_pipe_kernel<pa::kE4, false><<<grid, pa::kPipeThreads, used, (cudaStream_t)stream>>>(
            table, ntensors, tiles, none, s, nonfinite, pa::kTile);
    return check_launch("adamw_step_pipe_kernel (no-alloc multi) launch");
}

// ===========================================================================
// Packed-E4 step over host-resident parameters, gradients and state
// ===========================================================================
// The tensors stay in (page-locked) host memory; the call streams them through
// a caller-provided device workspace in chunks.  Three stages rotate: while
// the step runs on chunk i (caller's stream), chunk i+1 is copied in (an
// internal upload stream) and chunk i-1 is copied out (an internal download
// stream); events order the three.  Each element crosses the host link as
// 12 bytes in (p, g, word) and 8 bytes out (p, word).
namespace {

constexpr int kHostStages = 3;

struct HostPipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t in_done[kHostStages] = {}, step_done[kHostStages] = {}, out_done[kHostStages] = {};
};

std::mutex g_pipe_mu;
HostPipe g_pipe[64];

pa_status host_pipe(int dev, HostPipe **out)
{
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming);
        for (int k = 0; k < kHostStages && e == cudaSuccess; ++k) {
            e = cudaEventCreateWithFlags(&hp.in_done[k], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&hp.step_done[k], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&hp.out_done[k], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return cuda_fail(e, "creating the host-step streams and events");
        hp.ready = true;
    }
    *out = &hp;
    return PA_OK;
}

// The device address of page-locked host memory mapped into the device's
// address space (cudaHostAlloc / cudaMallocHost / cudaHostRegister), or false.
bool device_view(const void *host, void **dev)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr)
        return false;
    *dev = a.devicePointer;
    return true;
}

// The step with the GPU reading and writing the mapped host arrays in place:
// every byte crosses the host link once (12 in, 8 out per parameter), both
// directions at once, with no copies and no staging in device memory.  The
// register-staged kernel (plain 16-byte loads and stores) is used: the bulk
// copies of the staged kernel are kept to device memory.
pa_status host_step_in_place(float *p, const float *g, uint32_t *state, int64_t n, int64_t step,
                             double lr, double beta1, double beta2, double eps, double wd,
                             unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    const pa_tensor t = {p, g, state, nullptr, n};
    Desc d;
    int64_t chunk = 0;
    if ((st = chunk_size(kSlotHostE4, n, &chunk)) != PA_OK)
        return st;
    const int64_t chunks = describe(t, pa::kE4, chunk, &d);
    d.chunk0 = 0;
    int grid = 0;
    if ((st = grid_for(kSlotHostE4, chunks, &grid)) != PA_OK)
        return st;
    if (s.bc2 == 1.0f)
        pa::adamw_step_kernel<pa::kE4, false, true, float><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(
            nullptr, 1, chunks, chunk, d, s, nonfinite);
    else
        pa::adamw_step_kernel<pa::kE4, false, false, float><<<grid, pa::kThreads, 0, (cudaStream_t)stream>>>(
            nullptr, 1, chunks, chunk, d, s, nonfinite);
    return check_launch("adamw_step_kernel (host memory in place) launch");
}

}  // namespace

extern "C" pa_status pa_adamw_step_packed_e4_host(float *p, const float *g, uint32_t *state,
                                                  int64_t n, int64_t step, double lr,
                                                  double beta1, double beta2, double eps,
                                                  double wd, void *workspace,
                                                  int64_t workspace_bytes,
                                                  unsigned long long *nonfinite,
                                                  pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (n < 0 || workspace_bytes < 0)
        return fail(PA_ERR_ARG, "n and workspace_bytes must be >= 0");
    if (n == 0)
        return ok();
    if (!p || !g || !state || !workspace)
        return fail(PA_ERR_NULL, "NULL pointer with n = %lld", (long long)n);
    if (!aligned(p, 4) || !aligned(g, 4) || !aligned(state, 4))
        return fail(PA_ERR_ALIGN, "host arrays must be 4-byte aligned");
    if (!aligned(workspace, 256))
        return fail(PA_ERR_ALIGN, "workspace must be 256-byte aligned");
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    // per stage: p, g, word arrays of `chunk` elements, each a multiple of 64
    int64_t chunk = workspace_bytes / (kHostStages * 12) / 64 * 64;
    if (chunk >= 65536) {
        void *dp = nullptr, *dg = nullptr, *ds = nullptr;
        if (device_view(p, &dp) && device_view(g, &dg) && device_view(state, &ds))
            return host_step_in_place(static_cast<float *>(dp), static_cast<const float *>(dg),
                                      static_cast<uint32_t *>(ds), n, step, lr, beta1, beta2, eps,
                                      wd, nonfinite, stream);
    }
    if (chunk < 65536)
        return fail(PA_ERR_ARG, "workspace of %lld bytes is below the minimum of %lld "
                    "(3 stages x 12 bytes x 65536 elements)", (long long)workspace_bytes,
                    (long long)(kHostStages * 12 * 65536));
    if (chunk > n)
        chunk = (n + 63) / 64 * 64;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_pipe_mu);  // one enqueue at a time per process
    HostPipe *hp = nullptr;
    if ((st = host_pipe(dev, &hp)) != PA_OK)
        return st;
    cudaStream_t cs = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    // uploads start after the work already queued on the caller's stream
    if ((e = cudaEventRecord(hp->entry, cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->up, hp->entry, 0)) != cudaSuccess)
        return cuda_fail(e, "ordering the host step after the caller's stream");
    const int64_t nchunks = (n + chunk - 1) / chunk;
    for (int64_t i = 0; i < nchunks; ++i) {
        const int k = (int)(i % kHostStages);
        const int64_t off = i * chunk, len = (n - off < chunk) ? n - off : chunk;
        float *sp = reinterpret_cast<float *>(ws + (size_t)k * 12 * chunk);
        float *sg = sp + chunk;
        uint32_t *sw = reinterpret_cast<uint32_t *>(sg + chunk);
        // the stage is free once its previous download has finished
        e = cudaStreamWaitEvent(hp->up, hp->out_done[k], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sp, p + off, (size_t)len * 4, cudaMemcpyHostToDevice, hp->up);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sg, g + off, (size_t)len * 4, cudaMemcpyHostToDevice, hp->up);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sw, state + off, (size_t)len * 4, cudaMemcpyHostToDevice, hp->up);
        if (e == cudaSuccess)
            e = cudaEventRecord(hp->in_done[k], hp->up);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(cs, hp->in_done[k], 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "host step upload");
        const pa_tensor t = {sp, sg, sw, nullptr, len};
        if ((st = step_single<pa::kE4>(t, step, lr, beta1, beta2, eps, wd, nonfinite, stream)) != PA_OK)
            return st;
        e = cudaEventRecord(hp->step_done[k], cs);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(hp->down, hp->step_done[k], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(p + off, sp, (size_t)len * 4, cudaMemcpyDeviceToHost, hp->down);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(state + off, sw, (size_t)len * 4, cudaMemcpyDeviceToHost, hp->down);
        if (e == cudaSuccess)
            e = cudaEventRecord(hp->out_done[k], hp->down);
        if (e != cudaSuccess)
            return cuda_fail(e, "host step download");
    }
    // the caller's stream resumes after the last downloads
    for (int k = 0; k < kHostStages; ++k)
        if ((e = cudaStreamWaitEvent(cs, hp->out_done[k], 0)) != cudaSuccess)
            return cuda_fail(e, "ordering the caller's stream after the host step");
    return ok();
}

// ===========================================================================
// Graph-replayable packed-E4 tensor-list step
// ===========================================================================
static_assert(sizeof(pa_hyper) == sizeof(pa::Scalars), "pa_hyper mirrors the kernel scalars");

extern "C" pa_status pa_hyper_table_fill(pa_hyper *rows, int64_t first_step, int32_t count,
                                         const double *lr_per_step, double lr, double beta1,
                                         double beta2, double eps, double wd, pa_stream stream)
{
    if (count < 0)
        return fail(PA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0)
        return ok();
    if (!rows)
        return fail(PA_ERR_NULL, "rows is NULL with count = %d", count);
    if (!aligned(rows, 16))
        return fail(PA_ERR_ALIGN, "rows must be 16-byte aligned");
    std::vector<Scalars> host((size_t)count);
    for (int32_t k = 0; k < count; ++k) {
        const double lrk = lr_per_step ? lr_per_step[k] : lr;
        pa_status st = make_scalars(first_step + k, lrk, beta1, beta2, eps, wd, &host[(size_t)k]);
        if (st != PA_OK)
            return st;
    }
    // pageable source: the copy returns once the rows have been staged
    cudaError_t e = cudaMemcpyAsync(rows, host.data(), (size_t)count * sizeof(Scalars),
                                    cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "uploading the scalar rows");
    return ok();
}

extern "C" pa_status pa_adamw_step_packed_e4_multi_graph(const pa_tensor *list, int32_t ntensors,
                                                         const pa_hyper *rows, int32_t nrows,
                                                         int64_t *index, int32_t *status,
                                                         unsigned long long *nonfinite,
                                                         pa_stream stream)
{
    if (ntensors < 0 || nrows < 0)
        return fail(PA_ERR_ARG, "ntensors and nrows must be >= 0");
    if (ntensors == 0)
        return ok();
    if (!list || !rows || !index)
        return fail(PA_ERR_NULL, "list, rows and index must not be NULL");
    if (!aligned(rows, 16) || !aligned(index, 8) || (status && !aligned(status, 4)))
        return fail(PA_ERR_ALIGN, "rows must be 16-byte, index 8-byte, status 4-byte aligned");
    pa_status st = check_counter(nonfinite);
    if (st != PA_OK)
        return st;
    int64_t total = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        if ((st = check_tensor(list[i], pa::kE4, i)) != PA_OK)
            return st;
        total += list[i].n;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    if (total > 0) {
        const Desc *table = nullptr;
        int64_t tiles = 0;
        if ((st = table_for(list, ntensors, pa::kE4, pa::kTile, &table, &tiles, 4, true)) != PA_OK)
            return st;
        const size_t smem = pa::PipeLayout<pa::kE4>::kBytes;  // the kernel's limit
        const size_t used = pa::PipeLayout<pa::kE4>::bytes_for(ntensors);
        int grid = 0;
        if ((st = pipe_grid((const void *)pa::adamw_step_table_kernel<pa::kE4>, smem, tiles, &grid)) !=
            PA_OK)
            return st;
        pa::adamw_step_table_kernel<pa::kE4><<<grid, pa::kPipeThreads, used, cs>>>(
            table, ntensors, tiles, reinterpret_cast<const Scalars *>(rows), nrows, index, status,
            nonfinite);
        if ((st = check_launch("adamw_step_table_kernel launch")) != PA_OK)
            return st;
    }
    pa::advance_index_kernel<<<1, 1, 0, cs>>>(index);
    return check_launch("advance_index_kernel launch");
}

// ===========================================================================
// Packed-E4 steps that read bfloat16 gradients
// ===========================================================================
extern "C" pa_status pa_adamw_step_packed_e4_bf16g(float *p, const uint16_t *g, uint32_t *state,
                                                   int64_t n, int64_t step, double lr,
                                                   double beta1, double beta2, double eps,
                                                   double wd, unsigned long long *nonfinite,
                                                   pa_stream stream)
{
    const pa_tensor t = {p, reinterpret_cast<const float *>(g), state, nullptr, n};
    return step_single<pa::kE4, __nv_bfloat16>(t, step, lr, beta1, beta2, eps, wd, nonfinite,
                                                stream);
}

extern "C" pa_status pa_adamw_step_packed_e4_multi_bf16g(const pa_tensor *list, int32_t ntensors,
                                                         int64_t step, double lr, double beta1,
                                                         double beta2, double eps, double wd,
                                                         unsigned long long *nonfinite,
                                                         pa_stream stream)
{
    return step_multi<pa::kE4, __nv_bfloat16>(list, ntensors, step, lr, beta1, beta2, eps, wd,
                                              nonfinite, stream);
}

// ===========================================================================
// Blockwise tensor-list step
// ===========================================================================
namespace {

struct BwTable {
    int device;
    std::vector<pa::BwDesc> host;
    pa::BwDesc *dev;
    int64_t items;  // work items of the staged kernel
    uint64_t last_use;
};

std::mutex g_bw_mu;
std::vector<BwTable> g_bw_tables;
uint64_t g_bw_tick = 0;

pa_status check_blockwise_tensor(const pa_blockwise_tensor &t, int index)
{
    if (t.n < 0)
        return fail(PA_ERR_ARG, "tensor %d: n must be >= 0 (got %lld)", index, (long long)t.n);
    if (t.n == 0)
        return PA_OK;
    if (!t.p || !t.g || !t.p_bf16 || !t.m_code || !t.m_absmax || !t.v_code || !t.v_absmax)
        return fail(PA_ERR_NULL, "tensor %d: NULL pointer with n = %lld", index, (long long)t.n);
    if (!aligned(t.p, 16) || !aligned(t.g, 16) || !aligned(t.p_bf16, 8) ||
        !aligned(t.m_code, 4) || !aligned(t.v_code, 4) || !aligned(t.m_absmax, 4) ||
        !aligned(t.v_absmax, 4))
        return fail(PA_ERR_ALIGN, "tensor %d: p, g 16-byte, p_bf16 8-byte, codes and absmax "
                    "4-byte alignment required", index);
    return PA_OK;
}

pa_status bw_table_for(const pa_blockwise_tensor *list, int32_t ntensors, const pa::BwDesc **out,
                       int64_t *items)
{
    std::vector<pa::BwDesc> host((size_t)ntensors);
    int64_t total = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        const pa_blockwise_tensor &t = list[i];
        host[(size_t)i].a = {t.p, t.g, t.p_bf16, t.m_code, t.m_absmax, t.v_code, t.v_absmax, t.n};
        host[(size_t)i].item0 = total;
        total += pa::bw_full_tiles(t.n) + (t.n % pa::kBlock != 0 ? 1 : 0);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_bw_mu);
    ++g_bw_tick;
    for (BwTable &t : g_bw_tables)
        if (t.device == dev && t.host.size() == host.size() &&
            std::memcmp(t.host.data(), host.data(), host.size() * sizeof(pa::BwDesc)) == 0) {
            t.last_use = g_bw_tick;
            *out = t.dev;
            *items = t.items;
            return PA_OK;
        }
    if (g_bw_tables.size() >= kMaxTables) {
        size_t old = 0;
        for (size_t k = 1; k < g_bw_tables.size(); ++k)
            if (g_bw_tables[k].last_use < g_bw_tables[old].last_use)
                old = k;
        int cur = dev;
        cudaSetDevice(g_bw_tables[old].device);
        cudaFree(g_bw_tables[old].dev);  // synchronises that device
        cudaSetDevice(cur);
        g_bw_tables.erase(g_bw_tables.begin() + (long)old);
    }
    BwTable t;
    t.device = dev;
    t.items = total;
    t.last_use = g_bw_tick;
    t.dev = nullptr;
    const size_t bytes = host.size() * sizeof(pa::BwDesc);
    if ((e = cudaMalloc((void **)&t.dev, bytes)) != cudaSuccess) {
        cudaGetLastError();
        return fail(PA_ERR_NOMEM, "cudaMalloc of a %zu-byte descriptor table: %s", bytes,
                    cudaGetErrorString(e));
    }
    if ((e = cudaMemcpy(t.dev, host.data(), bytes, cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(t.dev);
        return cuda_fail(e, "descriptor table upload");
    }
    t.host = std::move(host);
    g_bw_tables.push_back(std::move(t));
    *out = g_bw_tables.back().dev;
    *items = g_bw_tables.back().items;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_adamw_step_blockwise8_multi(const pa_blockwise_tensor *list,
                                                    int32_t ntensors, const float *qmap1,
                                                    const float *qmap2, int64_t step, double lr,
                                                    double beta1, double beta2, double eps,
                                                    double wd, unsigned long long *nonfinite,
                                                    pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (ntensors < 0)
        return fail(PA_ERR_ARG, "ntensors must be >= 0 (got %d)", ntensors);
    if (ntensors == 0)
        return ok();
    if (!list || !qmap1 || !qmap2)
        return fail(PA_ERR_NULL, "list and maps must not be NULL");
    if (!aligned(qmap1, 4) || !aligned(qmap2, 4))
        return fail(PA_ERR_ALIGN, "maps must be 4-byte aligned");
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    int64_t total = 0;
    for (int32_t i = 0; i < ntensors; ++i) {
        if ((st = check_blockwise_tensor(list[i], i)) != PA_OK)
            return st;
        total += list[i].n;
    }
    if (total == 0)
        return ok();
    const pa::BwDesc *table = nullptr;
    int64_t items = 0;
    if ((st = bw_table_for(list, ntensors, &table, &items)) != PA_OK)
        return st;
    int grid = 0;
    if ((st = pipe_grid((const void *)pa::blockwise8_pipe_kernel<true>, pa::kBwSmemBytes, items,
                        &grid, pa::kBwThreads)) != PA_OK)
        return st;
    pa::BwDesc none;
    std::memset(&none, 0, sizeof none);
    pa::blockwise8_pipe_kernel<true><<<grid, pa::kBwThreads, pa::kBwSmemBytes, (cudaStream_t)stream>>>(
        table, ntensors, items, none, qmap1, qmap2, s, nonfinite);
    return check_launch("blockwise8_pipe_kernel (multi) launch");
}

pa_status release_blockwise_tables()
{
    std::lock_guard<std::mutex> lock(g_bw_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (BwTable &t : g_bw_tables) {
        cudaSetDevice(t.device);
        cudaFree(t.dev);
    }
    g_bw_tables.clear();
    cudaSetDevice(cur);
    return PA_OK;
}

// ===========================================================================
// TurboAdam-style step (UState first moment, 1Q second moment)
// ===========================================================================
extern "C" pa_status pa_turbo_step(float *p, const float *g, int64_t n, const pa_turbo_state *state,
                                   int64_t step, double lr, double beta1, double beta2, double eps,
                                   double wd, double m_step_factor, uint64_t seed,
                                   unsigned long long *nonfinite, pa_stream stream)
{
    Scalars s;
    pa_status st = make_scalars(step, lr, beta1, beta2, eps, wd, &s);
    if (st != PA_OK)
        return st;
    if (!(beta1 * beta1 < beta2))
        return fail(PA_ERR_ARG, "UState needs beta1^2 < beta2 (got %g, %g)", beta1, beta2);
    if (!std::isfinite(m_step_factor) || !(m_step_factor > 0.0))
        return fail(PA_ERR_ARG, "m_step_factor must be finite and > 0 (got %g)", m_step_factor);
    if (n < 0)
        return fail(PA_ERR_ARG, "n must be >= 0 (got %lld)", (long long)n);
    if (n > ((int64_t)1 << 40) || step >= ((int64_t)1 << 22))
        return fail(PA_ERR_ARG, "n must be <= 2^40 and step < 2^22 (the rounding counter's fields)");
    if (n == 0)
        return ok();
    if (!state)
        return fail(PA_ERR_NULL, "state is NULL");
    const pa_turbo_state t = *state;
    if (!p || !g || !t.ucode || !t.umean || !t.uscal || !t.vidx || !t.vend)
        return fail(PA_ERR_NULL, "NULL pointer with n = %lld", (long long)n);
    if (!aligned(p, 16) || !aligned(g, 16))
        return fail(PA_ERR_ALIGN, "p and g must be 16-byte aligned");
    if (!aligned(t.umean, 2) || !aligned(t.vidx, 2) || !aligned(t.vend, 2) || !aligned(t.uscal, 4))
        return fail(PA_ERR_ALIGN, "umean, vidx, vend must be 2-byte and uscal 4-byte aligned");
    if ((st = check_counter(nonfinite)) != PA_OK)
        return st;
    pa::TurboArgs a = {p, g, n, t.ucode, t.umean, t.uscal, t.vidx, t.vend};
    pa::TurboScalars ts;
    ts.s = s;
    ts.bc1 = (float)(1.0 - std::pow(beta1, (double)step));
    ts.bc1p = (float)(1.0 - std::pow(beta1, (double)(step - 1)));
    ts.bc2p = (float)(1.0 - std::pow(beta2, (double)(step - 1)));
    ts.seed = seed;
    ts.step = step;
    const int64_t blocks = (n + pa::kTurboBlock - 1) / pa::kTurboBlock;
    int grid = 0;
    if ((st = grid_for(kSlotTurbo, (blocks + pa::kTurboWarps - 1) / pa::kTurboWarps, &grid)) != PA_OK)
        return st;
    cudaStream_t cs = (cudaStream_t)stream;
    pa::turbo_step_kernel<<<grid, pa::kTurboThreads, 0, cs>>>(a, ts, nonfinite);
    if ((st = check_launch("turbo_step_kernel launch")) != PA_OK)
        return st;
    pa::turbo_finalize_kernel<<<1, 32, 0, cs>>>(t.uscal, (float)n, (float)m_step_factor);
    return check_launch("turbo_finalize_kernel launch");
}
