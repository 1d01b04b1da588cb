/*
 * bitlinear.h - C ABI of the B300 (sm_103a) BitNet b1.58 BitLinear library.
 *
 * The BitLinear layer of BitNet b1.58 (cheatsheet.md, "BitNet b1.58とは？")
 * replaces a linear layer: weights are ternary {-1, 0, +1}, obtained by
 * scaling with their mean absolute value and rounding; activations are
 * 8-bit, scaled per token.  asi.tokyo, "マイクロソフトが偶然に作った史上最も
 * 効率的なAI" (2025-04-27), in the paragraph on running the model on a GPU,
 * describes a kernel that packs four ternary weights per byte and unpacks
 * them next to the math units before multiplying with 8-bit activations.  This library
 * is that path, written for one B300:
 *
 *   bitlinear_pack_weights   fp32 W -> gamma = mean|W| (exact) + packed 2-bit codes
 *   bitlinear_pack_ternary   int8 Wq in {-1,0,1} -> packed 2-bit codes
 *   bitlinear_quant_act      bf16 x -> RMSNorm + per-token absmax int8 q, token scale
 *   bitlinear_forward        q x packed W -> exact int32 -> rescaled bf16 out
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     the library never frees or retains them past the call's stream work.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All calls are asynchronous with respect to the host: they
 *     enqueue kernels and return.  No call synchronises the device.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid argument returns BITLINEAR_ERR_INVALID_ARG and enqueues nothing.
 *   - A failed kernel launch returns BITLINEAR_ERR_CUDA.
 *   - No exception crosses this boundary and nothing is printed (except the
 *     debug build's report of a failed bounds check, on stderr).
 *   - Matrices are row-major.  W is [N out, K in] (K contiguous); x, q are
 *     [M tokens, K]; out, acc are [M, N].
 *   - K must be a multiple of 16 (so every row starts on a 16-byte
 *     boundary); N >= 1, M >= 0 (M = 0 is a no-op).  Device pointers must be
 *     16-byte aligned, except the scalar/vector ones noted (4-byte).
 *
 * Packed weight layout (shared by both matmul engines).  Np = 16*ceil(N/16),
 * Kp = 128*ceil(K/128).  The buffer is Np*Kp/4 bytes of 2-bit codes
 * (code = Wq + 1: 00 = -1, 01 = 0, 10 = +1; 11 never written).  It is made
 * of 512-byte tiles, one per (row group r = n/16, k block c = k/128), tile
 * index r*(Kp/128) + c.  Inside a tile, with i = n%16, kk = k%128:
 *   g = i%8, u = i/8, t = kk/32, j = kk%32,
 *   P = j/16, m = (j%16)/4, sb = (j%4)/2, h = j%2, p = 2m + sb,
 *   byte = 16*(4g + t) + 4*(2P + u) + (16h + 2p)/8,  shift = (16h + 2p)%8.
 * So the 16 bytes at 16*(4g+t) hold rows g and g+8 of the group over
 * k in [32t, 32t+32), one 32-bit word per (row, 16-k half).  Padding
 * positions (n >= N or k >= K) hold code 01.  The byte format is stable: a
 * caller may save and reload packed buffers.
 */
#ifndef BITLINEAR_H_
#define BITLINEAR_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BITLINEAR_API __attribute__((visibility("default")))
#else
#define BITLINEAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BITLINEAR_OK = 0,
    BITLINEAR_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or stream */
    BITLINEAR_ERR_UNSUPPORTED = 2, /* no sm_103a device / shape beyond limits */
    BITLINEAR_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    BITLINEAR_ERR_TIMEOUT = 4,     /* a kernel gave up a bounded wait */
    BITLINEAR_ERR_STATE = 5,       /* a pending factor buffer was produced into again */
    BITLINEAR_ERR_BOUNDS = 6       /* debug build: a device bounds check failed */
} bitlinear_status_t;

/* Static, NUL-terminated description of a status code (never NULL). */
BITLINEAR_API const char *bitlinear_status_string(int status);

/* Library ABI version (major*100 + minor).  1.01 added
 * bitlinear_set_fused_prepass, bitlinear_debug_selftest and
 * BITLINEAR_ERR_BOUNDS; every 1.00 entry point is unchanged. */
BITLINEAR_API int bitlinear_version(void);

/* Bytes of the packed buffer for an [N, K] weight matrix:
 * 16*ceil(N/16) * 128*ceil(K/128) / 4.  Returns 0 if N < 1 or K < 1. */
BITLINEAR_API size_t bitlinear_packed_bytes(int64_t N, int64_t K);

/*
 * Absmean ternarisation and packing of fp32 master weights
 * (cheatsheet.md "BitNet b1.58とは？": weights scaled by their mean
 * absolute value, rounded to the nearest integer in {-1,0,+1};
 * asi.tokyo: four weights per byte).
 *
 *   gamma = (float)( round_to_double( sum_{n,k} |W[n,k]| ) / (N*K) )
 *           where the sum is exact (order independent) and rounded once;
 *   Wq    = clamp(rint_half_even( W / (gamma + eps) ), -1, 1)
 *           with fp32 add and fp32 divide, each correctly rounded.
 *
 *   W        device, fp32 [N, K] row-major, 16-byte aligned, finite values
 *            (non-finite values give an unspecified gamma and codes, and no
 *            fault).
 *   eps      added to gamma before dividing (1e-5 in the workloads).
 *   packed   device, bitlinear_packed_bytes(N, K) bytes, 16-byte aligned;
 *            fully overwritten (padding included).
 *   gamma    device, one float, 4-byte aligned; written by the device.
 *   stream   see conventions.
 * Uses a small per-device workspace (256 64-bit counters) that the library
 * allocates on the first call on each device and keeps until process exit;
 * that first call is therefore not capturable in a CUDA graph.  Calls on
 * different streams of the same device must not overlap in time.
 * Errors: INVALID_ARG (null/misaligned pointer, N < 1, K < 1, K % 16 != 0),
 * UNSUPPORTED (N*K > 2^40 weights: the exact 64-bit bucket sums could
 * overflow), CUDA (workspace allocation or launch failure).
 */
BITLINEAR_API bitlinear_status_t bitlinear_pack_weights(const float *W, int64_t N, int64_t K, float eps,
                                          uint8_t *packed, float *gamma, void *stream);

/*
 * Same result as bitlinear_pack_weights, for callers that cannot allocate
 * device memory: code whose device memory is all owned by another allocator
 * (a serving runtime's arena or pool), or code that must not take the
 * driver's allocation lock at that point.  This entry point allocates
 * nothing; the pages have no counterpart for it.
 *
 * Its scratch is a fixed device array of 256 64-bit counters (2 KB) built
 * into the library, present on every GPU that loads the library until the
 * process exits.  Limit: N*K <= 2^40 weights (each counter then stays below
 * 2^64); larger matrices return BITLINEAR_ERR_UNSUPPORTED.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call clears and reuses the same array,
 * so calls that overlap on the GPU (other streams, other threads) race and
 * give wrong results: serialise them.
 * Arguments, layout and other errors as bitlinear_pack_weights.
 */
BITLINEAR_API bitlinear_status_t bitlinear_pack_weights_noalloc(const float *W, int64_t N,
                                                                int64_t K, float eps,
                                                                uint8_t *packed, float *gamma,
                                                                void *stream);

/*
 * Packing of weights that are already ternary (the scale gamma is kept by
 * the caller).  Wq: device int8 [N, K] with values in {-1, 0, +1}
 * (other values are clamped to that range).  packed as above.
 * Errors: INVALID_ARG (null/misaligned pointer, N < 1, K < 1, K % 16 != 0).
 */
BITLINEAR_API bitlinear_status_t bitlinear_pack_ternary(const int8_t *Wq, int64_t N, int64_t K,
                                          uint8_t *packed, void *stream);

/*
 * Fused RMSNorm + per-token absmax int8 quantisation of activations
 * (cheatsheet.md "BitNet b1.58とは？": activations scaled per token to
 * 8 bits; RMSNorm from the LLaMA parts; lumen-it.ai: absmax quantisation).
 * For each token m, with v_k = x[m,k] * gain[k] (fp32; gain = 1 if NULL):
 *   mx   = max(max_k |v_k|, 1e-5f)
 *   c    = 127.0f / mx                              (fp32 divide)
 *   q_k  = clamp(rint_half_even(v_k * c), -128, 127) (fp32 multiply)
 *   r    = 1 / sqrt(sum_k v_k^2 / K + eps)          (double)
 *   tok_scale[m] = (float)(r * mx / 127)
 * RMSNorm's factor r > 0 cancels inside absmax, so q depends only on v;
 * q * tok_scale approximates RMSNorm(x) * gain to half a quantisation step.
 *
 *   x_bf16     device, bf16 [M, K], 16-byte aligned.
 *   gain_bf16  device, bf16 [K] or NULL, 16-byte aligned.
 *   q          device, int8 [M, K], 16-byte aligned.
 *   tok_scale  device, fp32 [M], 4-byte aligned.
 * q is bit-exact (no float reduction decides it); tok_scale is computed
 * with compensated fp32 sums and correctly rounded fp32 steps, within a few
 * 1e-7 relative of the double-precision definition above.
 * Errors: INVALID_ARG (null/misaligned pointer, M < 0, K < 16, K % 16 != 0).
 */
BITLINEAR_API bitlinear_status_t bitlinear_quant_act(const void *x_bf16, const void *gain_bf16, int64_t M,
                                       int64_t K, float eps, int8_t *q, float *tok_scale,
                                       void *stream);

/*
 * The BitLinear matmul (asi.tokyo: packed weights are unpacked next to
 * the math units and multiplied with 8-bit blocks; cheatsheet.md: the
 * matmul reduces to additions):
 *   acc[m,n] = sum_k q[m,k] * Wq[n,k]                  (exact int32)
 *   out[m,n] = bf16_rne( (float)acc[m,n] * (gamma * tok_scale[m]) )
 *              (gamma * tok_scale[m] is one fp32 multiply, then one fp32
 *              multiply by the accumulator, then round-to-nearest-even)
 *
 *   q          device, int8 [M, K] from bitlinear_quant_act, 16-byte aligned.
 *   tok_scale  device, fp32 [M], 4-byte aligned.
 *   packed     device, packed weights of an [N, K] matrix.
 *   gamma      device, one float (the weight scale), 4-byte aligned.
 *   out_bf16   device, bf16 [M, N], 16-byte aligned.
 *   acc_out    device, int32 [M, N], 16-byte aligned, or NULL (the exact
 *              integer accumulators, for checking).
 * Weights are static, so the kernels start reading `packed` before they
 * wait for the kernel that precedes them in the stream (the loads overlap
 * that kernel).  `packed` must therefore be final when this call's work
 * starts: it is when it was written by bitlinear_pack_weights /
 * bitlinear_pack_ternary or by a copy (cudaMemcpy*) earlier in the stream,
 * or by anything on another stream joined to this one with
 * cudaStreamWaitEvent.  Do not write it with a kernel of your own launched
 * immediately before this call on the same stream: launch that kernel on
 * another stream and join the streams with an event instead.
 * Engine choice is internal (bitlinear_set_engine overrides it): up to 32
 * tokens, up to 48 unless K >= 8192, N <= K and N*K >= 2^24, and up to 64
 * where K < 6912 or N*K < 2^24, the decode GEMV (legacy tensor MMA on
 * register-unpacked codes; above 16 tokens in 16-token chunks of one
 * launch); otherwise the tcgen05 GEMM (TMEM accumulators), with its K range
 * split across a cluster where the output tiles alone would leave most SMs
 * idle.  Above 256 tokens, and above 32 for matrices of at least 2^24
 * weights, the int8 activations are first widened to f16
 * (exact) into a buffer taken, stream-ordered, from a
 * memory pool the library keeps per device (M*K*2 bytes, returned to the
 * pool at the end of the call; the pool keeps its memory for later calls).
 * All engines give identical results.
 * Every bounded wait inside the GEMM that expires sets a device status
 * word; bitlinear_check_status reports it.
 * Errors: INVALID_ARG (null/misaligned pointer, M < 0, N < 1, K < 16,
 * K % 16 != 0, K > 65536: the fp32 tensor-core sums stay exact below
 * that), UNSUPPORTED (more than 65535*64 tokens, or more than 65535*4 row
 * groups on the GEMV), CUDA (launch failure, or the widening buffer could
 * not be allocated; the runtime's last-error state is cleared, so the
 * failure is reported here only).
 */
BITLINEAR_API bitlinear_status_t bitlinear_forward(const int8_t *q, const float *tok_scale,
                                     const uint8_t *packed, const float *gamma, int64_t M,
                                     int64_t N, int64_t K, void *out_bf16, int32_t *acc_out,
                                     void *stream);

/*
 * bitlinear_quant_act with the quantised activations stored as f16 (their
 * exact integer values, -128..127) instead of int8, for
 * bitlinear_forward_f16.  Same q values and token scales as
 * bitlinear_quant_act; q_f16: device f16 [M, K], 16-byte aligned.
 * Errors as bitlinear_quant_act.
 */
BITLINEAR_API bitlinear_status_t bitlinear_quant_act_f16(const void *x_bf16, const void *gain_bf16,
                                                         int64_t M, int64_t K, float eps, void *q_f16,
                                                         float *tok_scale, void *stream);

/*
 * bitlinear_forward for f16 activations from bitlinear_quant_act_f16, any
 * M >= 1: always the tensor-core GEMM (split across a cluster at small
 * tile counts), which loads the activation tiles by tensor-map copy
 * straight into the layout its MMAs read.  It keeps the GEMM below 64
 * tokens too: measured on the 2B shapes with weights from HBM, 7.5-11.5 us
 * at 32-64 tokens against 6.2-13.5 us for bitlinear_forward (the GEMV
 * there), within 20 % either way, and the decode GEMV reads int8
 * activations only.  Identical results to bitlinear_forward on the same
 * values; the same weight contract.
 * Errors: as bitlinear_forward.
 */
BITLINEAR_API bitlinear_status_t bitlinear_forward_f16(const void *q_f16, const float *tok_scale,
                                                       const uint8_t *packed, const float *gamma,
                                                       int64_t M, int64_t N, int64_t K, void *out_bf16,
                                                       int32_t *acc_out, void *stream);

/*
 * Fused decode path (M <= 16): the activation quantiser folded into the
 * decode GEMV (cheatsheet.md "BitNet b1.58とは？": every BitLinear input is
 * quantised per token by its absolute maximum and rescaled by its RMS).
 *
 * A "factor buffer" (bitlinear_fused_stats_bytes() bytes, device, 16-byte
 * aligned) travels with an activation matrix [M, K] in bf16.  It yields each
 * token's c = 127 / max(max_k |v|, 1e-5) and tok_scale = rms^-1 * max / 127
 * (rms = sqrt(sum v^2 / K + eps)), either as published values or as a
 * pending accumulator filled by the launch that produced the activation.
 * Zero a factor buffer once (cudaMemset) before its first use.
 *
 *   bitlinear_act_stats       publishes the factors of an input x (bf16
 *                             [M, K]) into stats, resetting any pending
 *                             state.
 *   bitlinear_forward_fused   for up to 4 projections j sharing the input x:
 *                             c and tok_scale from x_stats, q = clamp(rint(
 *                             x * c), -128, 127) (bit-identical to
 *                             bitlinear_quant_act), acc = sum q * Wq (exact
 *                             int32), out_j = bf16(acc * (gamma_j *
 *                             tok_scale)); and, if stats_j is given, out_j's
 *                             max |v| and sum v^2 per token accumulated into
 *                             stats_j, which becomes pending.  The launch
 *                             consumes x_stats: if it was pending, its
 *                             factors are published and its accumulator
 *                             cleared by the time the launch ends.  The sums
 *                             of squares use fp32 atomics (order varies):
 *                             token scales agree with the definition to about
 *                             1e-7, and every CTA of the consuming launch
 *                             uses the same bits.
 *   bitlinear_fused_factors   copies the factors of a factor buffer for
 *                             [M, K] to c_out / ts_out (device fp32 [M] each,
 *                             either may be NULL); with consume != 0 it also
 *                             publishes them and clears a pending
 *                             accumulator, like a consuming launch.
 * A pending factor buffer must be consumed (by bitlinear_forward_fused or
 * bitlinear_fused_factors with consume) or reset (bitlinear_act_stats)
 * before it is produced into again; producing into a pending buffer sets the
 * status word, which bitlinear_check_status reports as
 * BITLINEAR_ERR_STATE.  x_stats must not be one of the stats_j, and the
 * stats_j must be distinct.  Weights follow the static-weight contract of
 * bitlinear_forward.  1 <= M <= 16, K % 16 == 0, K <= 65536.
 * Errors: INVALID_ARG (sizes, pointers, alignment, shared buffers),
 * UNSUPPORTED (too many row blocks), CUDA.
 */
typedef struct {
    const uint8_t *packed;  /* device: packed weights of an [N, K] matrix */
    const float *gamma;     /* device: its scale (one float) */
    int64_t N;              /* output features, 1 <= N <= 2^24 */
    void *out_bf16;         /* device bf16 [M, N], 16-byte aligned */
    int32_t *acc_out;       /* device int32 [M, N] or NULL (exact accumulators) */
    void *stats;            /* device factor buffer for out, or NULL */
} bitlinear_fused_proj_t;

BITLINEAR_API size_t bitlinear_fused_stats_bytes(void);
BITLINEAR_API bitlinear_status_t bitlinear_act_stats(const void *x_bf16, int64_t M, int64_t K, float eps,
                                                     void *stats, void *stream);
BITLINEAR_API bitlinear_status_t bitlinear_forward_fused(const void *x_bf16, void *x_stats,
                                                         int64_t M, int64_t K, int32_t nproj,
                                                         const bitlinear_fused_proj_t *projs, float eps,
                                                         void *stream);
BITLINEAR_API bitlinear_status_t bitlinear_fused_factors(void *stats, int64_t M, int64_t K, float eps,
                                                         int32_t consume, float *c_out, float *ts_out,
                                                         void *stream);

/*
 * How bitlinear_forward_fused quantises its input.  Below the threshold
 * (packed weight bytes of the launch: sum over j of the packed size of
 * projection j, rounded up to 64-row blocks) every CTA quantises the slice
 * of x it reads; at or above it, one pre-pass kernel quantises x into
 * stream-ordered scratch memory (M * K bytes, from a library-owned pool) and
 * the GEMV reads int8.  Same bits either way: the choice changes only the
 * time.  min_weight_bytes: -1 restores the default (16 MiB, measured: the
 * 70B stack at one token takes 8.28 ms without the pre-pass and 7.32 with
 * it from 16 MiB; the 3B stack's launches, all under 14 MB, are 6 % slower
 * with it), 0 uses the pre-pass always, larger values
 * set the threshold.  Process-wide, not per stream.  Errors: INVALID_ARG
 * (below -1).  With the pre-pass, bitlinear_forward_fused can also return
 * CUDA when the scratch allocation fails (nothing is launched then).
 */
BITLINEAR_API bitlinear_status_t bitlinear_set_fused_prepass(int64_t min_weight_bytes);

/*
 * Reads and clears the current device's kernel status word after
 * synchronising `stream`.  Returns BITLINEAR_OK, BITLINEAR_ERR_BOUNDS
 * (debug build, below), BITLINEAR_ERR_STATE (a
 * pending factor buffer was produced into again), BITLINEAR_ERR_TIMEOUT (a
 * bounded wait gave up), or BITLINEAR_ERR_CUDA if the stream reports an
 * error.
 */
BITLINEAR_API bitlinear_status_t bitlinear_check_status(void *stream);

/*
 * Debug build.  Compiled with -DBITLINEAR_DEBUG (libbitlinear_debug.so,
 * `python bitlinear_02_b300/build.py --debug`), every plain global load and
 * store of the kernels first checks its offset against its buffer's extent;
 * a failed check skips the access and is recorded (no trap: the context
 * stays usable).  bitlinear_check_status then returns BITLINEAR_ERR_BOUNDS
 * (before any other code) and names the source file and check sites on
 * stderr.  Tensor-map copies are bounds-checked by the hardware.  Release
 * builds carry no checks.
 * bitlinear_debug_selftest enqueues a kernel that records one failed check
 * without touching memory, to exercise that reporting path; release builds
 * return BITLINEAR_ERR_UNSUPPORTED and enqueue nothing.
 */
BITLINEAR_API bitlinear_status_t bitlinear_debug_selftest(void *stream);

/*
 * Test hook: sets the spin limit of every bounded wait in the library's
 * kernels (iterations of a try-wait loop; 0 restores the default).  A tiny
 * limit makes the waits give up, so the timeout path can be exercised
 * without hanging or faulting the GPU.
 */
BITLINEAR_API void bitlinear_set_wait_limit(uint32_t iterations);

/*
 * Engine choice of bitlinear_forward and bitlinear_forward_f16 (tuning and
 * testing; the defaults are measured choices, and every setting computes the
 * same bits).
 *   gemv_max_tokens: batches of up to this many tokens run bitlinear_forward
 *     on the decode GEMV engine (16-token chunks of one launch), larger ones
 *     on the tensor-core GEMM; 0 sends every batch to the GEMM; at most 64.
 *     -1 restores the default: the GEMV up to 32 tokens; at 33-48 tokens too
 *     unless K >= 8192, N <= K and N*K >= 2^24, and at 49-64 tokens unless
 *     K >= 6912 and N*K >= 2^24 (where the split-K GEMM on widened
 *     activations was measured faster).
 *   split_k: CTAs per cluster that share one GEMM output tile's k range
 *     (their int32 partial tiles summed through distributed shared memory).
 *     0 restores the default (the planner picks 1..16 from the tile count,
 *     the SM count and K); 1..16 forces that value where K has at least that
 *     many 64-k stages.
 * Returns BITLINEAR_ERR_INVALID_ARG for a value out of range (nothing
 * changes), else BITLINEAR_OK.  Settings are process-wide.
 */
BITLINEAR_API bitlinear_status_t bitlinear_set_engine(int32_t gemv_max_tokens, int32_t split_k);

/* ---------------------------------------------------------------------
 * Variant weight formats (decode engines, M <= 64 tokens).
 *
 * Five ternary digits per byte (vi.news.hada.io topic 20406, the comments
 * on ternary packing: 3^5 = 243 <= 256, so a b1.58 weight needs 1.6 bits
 * rather than 2).  Digits e = Wq + 1, most significant first, form
 * v = e0*81 + e1*27 + e2*9 + e3*3 + e4, stored as b = ceil(256 v / 243).
 * Layout: Np = 16*ceil(N/16), K5 = 160*ceil(K/160); Np*K5/5 bytes in
 * 512-byte tiles, one per (row group r = n/16, k block c = k/160), tile
 * index r*(K5/160) + c.  Inside a tile, with i = n%16, kk = k%160:
 *   g = i%8, u = i/8, t = kk/40, j = (kk%40)/5, d = kk%5,
 *   byte 16*(4g + t) + 8u + j of the tile holds digit d of (n, k).
 * Padding positions hold digit 1 (weight 0).
 */

/* Bytes of the five-digit layout for an N x K matrix (0 if N or K < 1). */
BITLINEAR_API size_t bitlinear_packed5_bytes(int64_t N, int64_t K);

/*
 * Re-encodes a 2-bit packed matrix (bitlinear_pack_weights /
 * bitlinear_pack_ternary output) into the five-digit layout, on the device.
 * packed: bitlinear_packed_bytes(N, K) bytes; packed5: caller-owned,
 * bitlinear_packed5_bytes(N, K) bytes; both 16-byte aligned device pointers.
 * The weight scale gamma is unchanged (bitlinear_forward5 takes it as is).
 * N >= 1, K >= 16, K % 16 == 0.  Errors: INVALID_ARG (shape, null or
 * misaligned pointer), UNSUPPORTED (more than 2^31 blocks of work), CUDA.
 */
BITLINEAR_API bitlinear_status_t bitlinear_repack5(const uint8_t *packed, int64_t N, int64_t K,
                                                   uint8_t *packed5, void *stream);

/*
 * bitlinear_forward on the five-digit layout: the same arguments, the same
 * int32 accumulators and bf16 outputs bit for bit, 20 % fewer weight bytes
 * read.  M <= 64 (the decode engine, 16-token chunks); larger M returns
 * UNSUPPORTED (the tensor-core GEMM reads the 2-bit layout).
 */
BITLINEAR_API bitlinear_status_t bitlinear_forward5(const int8_t *q, const float *tok_scale,
                                                    const uint8_t *packed5, const float *gamma,
                                                    int64_t M, int64_t N, int64_t K, void *out_bf16,
                                                    int32_t *acc_out, void *stream);

/*
 * The original 1-bit BitNet (lumen-it.ai BitNet article: weights binarised
 * to +1 / -1 by the signum function, absmax activations, quantisation in
 * groups).  Wb = +1 where W > 0, -1 elsewhere (zero goes to -1); the N rows
 * form G groups of N/G consecutive rows, each with its own scale
 * beta_g = mean |W| over the group (exact sum rounded once, as gamma);
 * out[m, n] = bf16(acc * (beta_{n / (N/G)} * tok_scale[m])),
 * acc = sum_k Wb[n, k] * q[m, k] exact.  Activations: bitlinear_quant_act.
 * Layout: Np = 16*ceil(N/16), K1 = 256*ceil(K/256); Np*K1/8 bytes in
 * 512-byte tiles, one per (r = n/16, c = k/256), tile index r*(K1/256) + c.
 * Inside a tile, with i = n%16, kk = k%256:
 *   g = i%8, u = i/8, t = kk/64, j = kk%64, P = j/32, s = (j%32)/4,
 *   sb = (j%4)/2, h = j%2, bit = 16h + 2s + sb,
 *   byte 16*(4g + t) + 4*(2P + u) + bit/8, bit bit%8 of it; 1 means +1.
 * Padding bits are 0.
 */
BITLINEAR_API size_t bitlinear_packed1_bytes(int64_t N, int64_t K);

/*
 * Binarises and packs fp32 W [N, K] (device, row-major, 16-byte aligned)
 * and writes the G group scales to beta[G] (device, 4-byte aligned).
 * packed1: caller-owned, bitlinear_packed1_bytes(N, K) bytes, 16-byte
 * aligned.  N % groups == 0, 1 <= groups <= 65536, K >= 16, K % 16 == 0,
 * N*K <= 2^40.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.  Uses the same 2 KB
 * device workspace as bitlinear_pack_weights.
 */
BITLINEAR_API bitlinear_status_t bitlinear_pack_binary(const float *W, int64_t N, int64_t K,
                                                       int64_t groups, uint8_t *packed1, float *beta,
                                                       void *stream);

/*
 * out = (Wb q) rescaled per group, as above.  q, tok_scale, out_bf16,
 * acc_out as in bitlinear_forward; beta: the groups scales (device, 4-byte
 * aligned).  M <= 64 (else UNSUPPORTED), N % groups == 0 (else
 * INVALID_ARG).
 */
BITLINEAR_API bitlinear_status_t bitlinear_forward_binary(const int8_t *q, const float *tok_scale,
                                                          const uint8_t *packed1, const float *beta,
                                                          int64_t groups, int64_t M, int64_t N, int64_t K,
                                                          void *out_bf16, int32_t *acc_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H_ */
