/*
 * packedadam.h -- C ABI of libpackedadam.so: the AdamW parameter update with
 * packed, quantized persistent moment state, as hand-written CUDA kernels for
 * NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   "Packed AdamW Reference" README v1.0.0, "The canonical format": one uint32
 *     state word per FP32 parameter; low 16 bits a signed finite E4M11 first
 *     moment m, high 16 bits an unsigned finite E4M12 uncorrected RMS
 *     r = sqrt(v); no shadow moments, block scales or stochastic rounding.
 *     The paragraph after it: gradients, bias correction, weight decay and the
 *     update are FP32; the new moments are used in FP32 and packed afterwards.
 *     Same page: FP32 AdamW and packed FP16-first/FP16-RMS comparison modes.
 *   "Packed AdamW / Reference / v1.0.0" code page, "Release scope" (decode,
 *     square the RMS, update in FP32, store afterwards; no conversion at the
 *     finite bound) and "Execution contract" (contiguous FP32 tensors on one
 *     device, a dense gradient every update, one global step).
 *   "TurboAdam" README, "The AdamW update remains AdamW": the recurrences.
 *   KBench "quantized-optimizer-state" reference.py, quantized_adamw_step and
 *     _requantise: the FP32 operation order and the 8-bit blockwise mode.
 *
 * Numerics (every entry point).  The host forms, in double and rounding once
 * to float: beta1, beta2, 1-beta1, 1-beta2, 1-beta2^step, lr/(1-beta1^step),
 * 1-lr*wd and eps.  Each element then computes, one IEEE binary32 rounding per
 * operation and no fused multiply-add:
 *     m' = beta1*m + (1-beta1)*g
 *     v' = beta2*v + ((1-beta2)*g)*g
 *     p' = p*(1-lr*wd) - ((lr/bc1)*m') / (sqrt(v'/bc2) + eps)
 * E4 lanes: IEEE-style layout without Inf/NaN codes, exponent bias 15 (E4M11
 * largest 2-2^-11, E4M12 largest 2-2^-12), subnormals kept, round to nearest
 * even, saturation at the largest finite value, NaN -> +0, the sign of zero
 * kept on the m lane, negative values -> 0 on the RMS lane.  FP16 lanes: IEEE
 * binary16, round to nearest even, saturation at +-65504, NaN -> +0.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers of the current CUDA device unless stated;
 *     the caller owns all memory and the stream.  Element counts are int64.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return after the launch.  Argument errors are found
 *     on the host before anything is launched.
 *   - `nonfinite` (nullable, device, 8-byte aligned): the number of elements
 *     whose new p, m or v is NaN or +-Inf is ADDED to *nonfinite.  Nothing is
 *     repaired: a NaN moment is stored as +0, an infinite one saturates.
 *   - n == 0 is a no-op returning PA_OK.  Buffers of one call must not overlap
 *     except where a parameter is updated in place.
 *   - Return value: PA_OK or an error code; pa_last_error() gives a one-line
 *     description of the most recent error on the calling thread.
 */
#ifndef PACKEDADAM_H
#define PACKEDADAM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pa_status;
#define PA_OK 0
#define PA_ERR_NULL 1  /* a required pointer is NULL while n > 0              */
#define PA_ERR_ARG 2   /* step < 1, beta outside [0,1), eps < 0, a non-finite
                          hyperparameter, n < 0, ntensors < 0, bad mode       */
#define PA_ERR_ALIGN 3 /* a pointer below its element alignment (see call)   */
#define PA_ERR_CUDA 4  /* a CUDA runtime call or launch failed                */
#define PA_ERR_NOMEM 5 /* the library could not allocate its descriptor table */

typedef void *pa_stream; /* cudaStream_t */

/* Library version, major*10000 + minor*100 + patch. */
int32_t pa_version(void);

/* Static name of a status code ("PA_OK", "PA_ERR_ARG", ...). */
const char *pa_status_string(pa_status status);

/* One-line description of the last error returned on this thread ("" if none). */
const char *pa_last_error(void);

/* ---------------------------------------------------------------------------
 * Packed-state codecs ("Packed AdamW Reference" README, "The canonical
 * format"; the README's inspect-formats command).
 *   pa_encode_state:  word[i] = E4M12(rms[i]) << 16 | E4M11(m[i])
 *   pa_decode_state:  m[i] = E4M11 value of the low 16 bits,
 *                     rms[i] = E4M12 value of the high 16 bits (exact)
 *   *_fp16 variants: the same with IEEE binary16 lanes (FP16-first/FP16-RMS).
 * Layout: m, rms float[n]; word uint32[n]; 4-byte aligned.  For encode,
 * `nonfinite` (nullable) counts elements with a non-finite m or rms.
 * ------------------------------------------------------------------------- */
pa_status pa_encode_state(const float *m, const float *rms, uint32_t *word, int64_t n,
                          unsigned long long *nonfinite, pa_stream stream);
pa_status pa_decode_state(const uint32_t *word, float *m, float *rms, int64_t n,
                          pa_stream stream);
pa_status pa_encode_state_fp16(const float *m, const float *rms, uint32_t *word, int64_t n,
                               unsigned long long *nonfinite, pa_stream stream);
pa_status pa_decode_state_fp16(const uint32_t *word, float *m, float *rms, int64_t n,
                               pa_stream stream);

/* ---------------------------------------------------------------------------
 * Single-tensor AdamW steps.  p (float[n]) and the state are updated in place;
 * g (float[n]) is read.  step is the 1-based global step.  All arrays 4-byte
 * aligned; when p, g and the state share their address modulo 16, the part
 * after up to 3 leading elements is staged through shared memory by bulk
 * copies (6144-element tiles, one CTA per SM, about 144 KB of shared memory;
 * 192 KB in the FP32 mode), otherwise elements are read with 4-byte accesses.
 * The staged kernels wait on their own copies with a 2-second limit; a wait
 * that runs out leaves that launch's results incomplete and is reported by
 * pa_device_fault (below), never by a hang.
 *
 * pa_adamw_step_packed_e4 -- the packed E4 step ("Packed AdamW / Reference /
 *   v1.0.0", "Release scope"): decode m and r from state[i], v = r*r, the FP32
 *   update, then state[i] = E4M12(sqrt(v')) << 16 | E4M11(m').
 * pa_adamw_step_packed_fp16 -- the same with binary16 lanes.
 * pa_adamw_step_fp32 -- ordinary AdamW with FP32 m and v (float[n] each).
 * ------------------------------------------------------------------------- */
pa_status pa_adamw_step_packed_e4(float *p, const float *g, uint32_t *state, int64_t n,
                                  int64_t step, double lr, double beta1, double beta2,
                                  double eps, double wd, unsigned long long *nonfinite,
                                  pa_stream stream);
pa_status pa_adamw_step_packed_fp16(float *p, const float *g, uint32_t *state, int64_t n,
                                    int64_t step, double lr, double beta1, double beta2,
                                    double eps, double wd, unsigned long long *nonfinite,
                                    pa_stream stream);
pa_status pa_adamw_step_fp32(float *p, const float *g, float *m, float *v, int64_t n,
                             int64_t step, double lr, double beta1, double beta2, double eps,
                             double wd, unsigned long long *nonfinite, pa_stream stream);

/* ---------------------------------------------------------------------------
 * 8-bit blockwise AdamW (KBench "quantized-optimizer-state" reference.py,
 * quantized_adamw_step and _requantise).  Blocks of 2048 consecutive
 * elements; nb = ceil(n / 2048) (the last block may be short and its absmax
 * covers its own elements only).
 *   m = qmap1[m_code[i]] * m_absmax[b],  v = qmap2[v_code[i]] * v_absmax[b]
 *   FP32 update as above; p_bf16[i] = bfloat16 round-to-nearest-even of p'.
 *   New m_absmax[b] = max |m'| over the block (NaN propagates), and
 *   m_code[i] = number of the 255 binary32 midpoints (qmap1[j]+qmap1[j+1])*0.5
 *   strictly below m' / max(absmax, 1e-30); likewise for v with qmap2.
 * p and g are read only (float[n], 16-byte aligned); p_bf16 uint16[n] (8-byte
 * aligned) receives the new parameters; m_code, v_code uint8[n] (4-byte
 * aligned) and m_absmax, v_absmax float[nb] are replaced in place; qmap1 and
 * qmap2 are ascending float[256] in device memory.
 * ------------------------------------------------------------------------- */
pa_status pa_adamw_step_blockwise8(const float *p, const float *g, uint16_t *p_bf16,
                                   uint8_t *m_code, float *m_absmax, uint8_t *v_code,
                                   float *v_absmax, const float *qmap1, const float *qmap2,
                                   int64_t n, int64_t step, double lr, double beta1,
                                   double beta2, double eps, double wd,
                                   unsigned long long *nonfinite, pa_stream stream);

/* Blockwise tensor-list step: pa_adamw_step_blockwise8 over every tensor of a
 * list in one persistent launch (blocks never span tensors: each tensor's
 * blocks start at its element 0).  list[t] (host, read during the call):
 * arrays as for pa_adamw_step_blockwise8 with n = list[t].n; both maps are
 * shared by the list.  The descriptor table is cached like the other lists'. */
typedef struct pa_blockwise_tensor {
    const float *p;
    const float *g;
    uint16_t *p_bf16;
    uint8_t *m_code;
    float *m_absmax;
    uint8_t *v_code;
    float *v_absmax;
    int64_t n;
} pa_blockwise_tensor;

pa_status pa_adamw_step_blockwise8_multi(const pa_blockwise_tensor *list, int32_t ntensors,
                                         const float *qmap1, const float *qmap2, int64_t step,
                                         double lr, double beta1, double beta2, double eps,
                                         double wd, unsigned long long *nonfinite,
                                         pa_stream stream);

/* ---------------------------------------------------------------------------
 * Multi-tensor steps: one persistent grid-stride launch over every tensor of
 * a list ("Packed AdamW / Reference / v1.0.0", "Execution contract", lists one
 * launch per tensor; this library replaces that with one launch per list).
 * The result equals the single-tensor call on each tensor.
 *
 * list[t] describes tensor t (host memory, read during the call only):
 *   p      float[n], updated in place
 *   g      float[n]
 *   state  uint32[n] (packed modes) or float m[n] (FP32 mode)
 *   state2 NULL (packed modes) or float v[n] (FP32 mode)
 * The library keeps a device copy of each distinct list of two or more
 * tensors it is given (its descriptor table, allocated with cudaMalloc on
 * first use of that list on the current device and reused while the list is
 * unchanged; at most 64 lists are kept, the least recently used is freed
 * first, except the lists of pa_adamw_step_packed_e4_multi_graph below, which
 * are kept until pa_release_tables).
 * pa_release_tables() frees them all; it synchronises the device.  A
 * one-tensor list is passed by value in the launch, like the single-tensor
 * calls: no table, no allocation, no copy, whatever its pointers.
 * ------------------------------------------------------------------------- */
typedef struct pa_tensor {
    float *p;
    const float *g;
    void *state;
    void *state2;
    int64_t n;
} pa_tensor;

pa_status pa_adamw_step_packed_e4_multi(const pa_tensor *list, int32_t ntensors, int64_t step,
                                        double lr, double beta1, double beta2, double eps,
                                        double wd, unsigned long long *nonfinite,
                                        pa_stream stream);
pa_status pa_adamw_step_packed_fp16_multi(const pa_tensor *list, int32_t ntensors,
                                          int64_t step, double lr, double beta1, double beta2,
                                          double eps, double wd, unsigned long long *nonfinite,
                                          pa_stream stream);
pa_status pa_adamw_step_fp32_multi(const pa_tensor *list, int32_t ntensors, int64_t step,
                                   double lr, double beta1, double beta2, double eps,
                                   double wd, unsigned long long *nonfinite, pa_stream stream);

/* ---------------------------------------------------------------------------
 * pa_adamw_step_packed_e4_multi_noalloc -- the step of
 * pa_adamw_step_packed_e4_multi (same arguments, same bits) for callers that
 * cannot have a library allocate device memory: for example a framework whose
 * caching allocator has reserved the device's memory and expects every
 * allocation to go through it, or a loop that must not meet the implicit
 * synchronisation of cudaMalloc and cudaFree.  The pages have no counterpart;
 * this entry point is an addition of this library.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  The list's
 * descriptor table goes into a fixed device array compiled into the library:
 * PA_NOALLOC_MAX_TENSORS = 1024 descriptors of 56 bytes, which every device
 * that loads the library holds until the process exits.  ntensors > 1024
 * returns PA_ERR_ARG.  The descriptors travel as the launch parameters of a
 * small kernel on `stream` (up to 512 per launch) that writes them into the
 * array ahead of the step kernel, so the call neither copies from host memory
 * nor waits for work already queued on `stream`.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls share the array and each rewrites the
 * part it uses: calls that overlap on the GPU (on different streams, or from
 * racing host threads) race on it.
 * ------------------------------------------------------------------------- */
pa_status pa_adamw_step_packed_e4_multi_noalloc(const pa_tensor *list, int32_t ntensors,
                                                int64_t step, double lr, double beta1,
                                                double beta2, double eps, double wd,
                                                unsigned long long *nonfinite,
                                                pa_stream stream);

/* ---------------------------------------------------------------------------
 * pa_adamw_step_packed_e4_host -- the packed E4 step (as pa_adamw_step_packed_e4)
 * over p, g and the state words held in HOST memory, for optimizer state kept
 * off the device ("Packed AdamW Reference" README, "The canonical format": the
 * state is 4 bytes per parameter instead of 8, which also shrinks the traffic
 * over the host link: 12 bytes in and 8 bytes out per parameter).
 * p, g, state: host arrays of n elements, 4-byte aligned.
 * When all three are page-locked and mapped into the device's address space
 * (cudaHostAlloc / cudaMallocHost / cudaHostRegister; torch's pin_memory), the
 * step kernel reads and writes them in place over the host link (one launch
 * on `stream`, both link directions at once, no copies; the workspace is
 * checked but not used).  Otherwise the call streams the arrays through the
 * workspace: page-locked memory lets those copies run asynchronously and
 * overlap, pageable memory works but copies synchronously.
 * workspace: caller-owned device memory, 256-byte aligned, of workspace_bytes
 * >= 3 * 12 * 65536 bytes; chunks of workspace_bytes / 36 elements (three
 * rotating stages), overlapping uploads, the step and downloads on two
 * internal streams (created on the first call on a device) and `stream`.
 * Either way the call returns after queueing and synchronising `stream` makes
 * the host arrays current.  Host enqueues are serialised by a process-wide
 * lock; the workspace and host arrays must not be touched until `stream` has
 * passed the call.  Errors as for the other steps; a workspace below the
 * minimum is PA_ERR_ARG, a misaligned one PA_ERR_ALIGN.
 * ------------------------------------------------------------------------- */
pa_status pa_adamw_step_packed_e4_host(float *p, const float *g, uint32_t *state, int64_t n,
                                       int64_t step, double lr, double beta1, double beta2,
                                       double eps, double wd, void *workspace,
                                       int64_t workspace_bytes, unsigned long long *nonfinite,
                                       pa_stream stream);

/* ---------------------------------------------------------------------------
 * Packed-E4 steps whose gradient is bfloat16 (uint16 bit patterns, 2-byte
 * aligned), as produced by mixed-precision backward passes: each gradient is
 * widened exactly to binary32 and the step is the packed E4 step above, bit for
 * bit.  The gradient costs 2 bytes instead of 4: 18 bytes per parameter.
 * The staged copies need the gradient 16-byte aligned where p's 16-byte body
 * starts (true for whole tensors from an allocator); a tensor without that is
 * updated with per-element accesses, with the same results.
 * pa_adamw_step_packed_e4_multi_bf16g reads list[t].g as a uint16 pointer.
 * ------------------------------------------------------------------------- */
pa_status pa_adamw_step_packed_e4_bf16g(float *p, const uint16_t *g, uint32_t *state, int64_t n,
                                        int64_t step, double lr, double beta1, double beta2,
                                        double eps, double wd, unsigned long long *nonfinite,
                                        pa_stream stream);
pa_status pa_adamw_step_packed_e4_multi_bf16g(const pa_tensor *list, int32_t ntensors,
                                              int64_t step, double lr, double beta1, double beta2,
                                              double eps, double wd, unsigned long long *nonfinite,
                                              pa_stream stream);

/* ---------------------------------------------------------------------------
 * Graph-replayable step.  pa_adamw_step_packed_e4_multi computes the step's
 * scalars on the host at every call, so a CUDA graph that captured it would
 * replay one step number forever.  Here the scalars come from a device table
 * of rows filled ahead of time and a device-side row index that the call
 * advances, so a captured call replays as consecutive steps with no host work.
 *
 * pa_hyper: the eight binary32 scalars of one step (formed as described at the
 * top of this header): beta1, beta2, 1-beta1, 1-beta2, 1-beta2^step,
 * lr/(1-beta1^step), 1-lr*wd, eps.
 * pa_hyper_table_fill: compute rows for steps first_step .. first_step+count-1
 *   and copy them to `rows` (device, 16-byte aligned, count entries) on
 *   `stream`; lr_per_step (host, count doubles, nullable) gives a schedule,
 *   otherwise `lr` is used for every row.  The host array is read during the
 *   call only.
 * pa_adamw_step_packed_e4_multi_graph: the packed E4 tensor-list step with the
 *   scalars of row *index (index: device int64), then *index += 1 (a second,
 *   one-thread launch on `stream`).  When *index is outside [0, nrows) nothing
 *   is updated and *status (device int32, nullable) is set to 1; the index
 *   still advances.  The list's descriptor table is made on the first call
 *   with that list (a cudaMalloc); make that first call before capturing, so a
 *   captured call finds it.  A captured launch holds that table's address, so
 *   the library keeps the table of every list given to this call, whatever
 *   other lists it sees later, until pa_release_tables or pa_shutdown, which
 *   free it: replaying a graph captured before either of them reads freed
 *   memory, so capture it again after them.  Results equal
 *   pa_adamw_step_packed_e4_multi at the same step and hyperparameters, bit
 *   for bit.
 * ------------------------------------------------------------------------- */
typedef struct pa_hyper {
    float b1, b2, c1, c2, bc2, ss, dk, ef;
} pa_hyper;

pa_status pa_hyper_table_fill(pa_hyper *rows, int64_t first_step, int32_t count,
                              const double *lr_per_step, double lr, double beta1, double beta2,
                              double eps, double wd, pa_stream stream);
pa_status pa_adamw_step_packed_e4_multi_graph(const pa_tensor *list, int32_t ntensors,
                                              const pa_hyper *rows, int32_t nrows, int64_t *index,
                                              int32_t *status, unsigned long long *nonfinite,
                                              pa_stream stream);

/* ---------------------------------------------------------------------------
 * TurboAdam-style step ("TurboAdam" README, turboadam 0.2.0, "How it works"):
 * the AdamW update from FP32 transient moments, with the first moment
 * persisted by UState (normalised Adam update units q = (m/(1-beta1^t)) /
 * (sqrt(v_persisted/(1-beta2^t)) + eps), a 2-bit four-level code per value, a
 * bf16 mean per 64 values, a one-step-lagged tensor scale) and the second
 * moment by 1Q (a 4-bit index per value on a logarithmic grid between two fp16
 * log endpoints per 128 values), both with stochastic rounding from a counter
 * hash.  One call: decode both states, rebuild the prior first moment in the
 * persisted second-moment frame, form m and v, update p in place, recompress
 * v, encode the next UState payload, then rotate the scales (the page's
 * "Fused CUDA path" and finaliser).  Readings where the page is silent (grid,
 * levels, hash, rounding, means) are stated in the library's design notes and
 * in csrc/turbo.cuh.
 *
 * pa_turbo_state (device arrays, caller-owned, all zero before the first step):
 *   ucode  uint8[(n+3)/4]        2-bit codes, element i at bits 2*(i%4) of byte i/4
 *   umean  uint16[(n+63)/64]     bf16 mean per 64 values
 *   uscal  float[3]              decode scale, encode scale, RMS accumulator
 *   vidx   uint8[(n+1)/2]        4-bit indices, element i in nibble i%2 of byte i/2
 *   vend   uint16[2*ceil(n/128)] fp16 endpoints (lo, hi) per 128 values
 * p, g: float[n], 16-byte aligned; umean, vidx and vend 2-byte aligned.
 * m_step_factor: the UState scale factor (1.1 on the page); seed: the
 * counter hash's seed (rounding for step t and element i depends only on
 * seed, t and i).  beta1^2 < beta2 is required (the page's finite coordinate
 * bound), else PA_ERR_ARG; so are step >= 2^22 and n > 2^40.  Other errors as
 * for the other steps.  The RMS accumulator is a parallel float sum, so the
 * next encode scale can differ from a sequential sum in its last bits (the
 * page says the same of its own CUDA path); everything else is exact.
 * ------------------------------------------------------------------------- */
typedef struct pa_turbo_state {
    uint8_t *ucode;
    uint16_t *umean;
    float *uscal;
    uint8_t *vidx;
    uint16_t *vend;
} pa_turbo_state;

pa_status pa_turbo_step(float *p, const float *g, int64_t n, const pa_turbo_state *state,
                        int64_t step, double lr, double beta1, double beta2, double eps, double wd,
                        double m_step_factor, uint64_t seed, unsigned long long *nonfinite,
                        pa_stream stream);

/* Device fault flag of the staged step kernels (current device): *code = 0
 * when no bounded wait has run out since the flag was last cleared, else 1 (the
 * copying warp found a stage still in use after 2 s), 2 (a copy had not landed
 * 2 s after the last tile) or 3 (a computing warp waited 2 s for a stage's
 * copies); the first fault is kept.  clear != 0 resets it to 0.  Synchronous:
 * the read waits for the work already queued on the legacy default stream.
 * PA_ERR_NULL if code is NULL. */
pa_status pa_device_fault(uint32_t *code, int32_t clear);

/* Frees every cached descriptor table on every device (synchronises them). */
pa_status pa_release_tables(void);

/* Releases what the library holds on the devices (the cached descriptor
 * tables); call it before unloading the library.  Later calls recreate what
 * they need. */
pa_status pa_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* PACKEDADAM_H */
