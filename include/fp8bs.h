/*
 * fp8bs -- small-M W8A8 FP8 block-scale linear for NVIDIA GB300 (sm_103a).
 *
 *   Y[M,N] = bf16( sum_kb ( sum_{k in kb} xq[m,k] * wq[n,k] ) * xs[m,kb] * ws[n/128,kb] )
 *
 * with the bf16 -> e4m3fn activation quantisation in 1x128 groups fused into
 * the same launch, and an optional power-of-two (ue8m0 / e8m0) scale variant.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "[AMD] Small-M FP8 block-scale GEMM with fused activation quant for
 *        gfx950 (Qwen3.5)", "Motivation" and "Modifications": one launch per
 *        linear for M <= 32; per-1x128-group activation quant from the row amax,
 *        bit-exact scales and fp8 bytes; the fp8 weight streamed once; one MMA
 *        per 128-wide K block followed by x_scale * w_scale in fp32; a cross-wave
 *        reduction to a bf16 output; a [N/128, K/128] fp32 weight scale; the
 *        support rules (bf16 input, 16-byte aligned rows, contiguous scales, no
 *        bias, no input scale).
 *   [P2] "[AMD] gfx950 small-batch MoE: expert-count gate for the small sort and
 *        FP8 block-scale small-M kernel", "Modifications": float8_e4m3fn weights
 *        with a 128x128 fp32 block scale applied to each partial sum.
 *   [P4] "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense 128x128 fp8
 *        linears (6/8)", "Motivation" and "Modifications": power-of-two 128x128
 *        weight scales kept as one e8m0 byte per block; ue8m0 per-1x128
 *        activation scales; an e8m0 operand must never be read as fp32.
 *
 * Conventions for every entry point:
 *   - Data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no memory, keeps no pointer after a call returns and never
 *     synchronises, except fp8bs_check_error and the first call of
 *     fp8bs_gemm_fused_static on each device (both documented there).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it; results are ready when it reaches them.
 *   - Return value: FP8BS_OK (0) or a negative fp8bs_status.  Argument faults
 *     are detected on the host, return at once and enqueue nothing.  Faults only
 *     the device can see (a packed weight of another shape or scale kind, a
 *     bounded wait that expired) are recorded in the workspace error word and
 *     reported by fp8bs_check_error.
 *   - Layouts are row-major.  bf16 values travel as uint16_t bit patterns and
 *     e4m3fn codes / e8m0 scale bytes as uint8_t.
 *   - e4m3fn: OCP FP8 E4M3 (bias 7, no infinities, largest finite 448).  Codes
 *     are round-to-nearest-even of x / scale, saturated to +-448, never NaN.
 *   - Scale kinds: FP8BS_SCALE_F32 stores fp32 scales; FP8BS_SCALE_UE8M0 stores
 *     one e8m0 byte b per scale, meaning 2^(b - 127).  The kind is always an
 *     explicit argument and is never inferred from the bytes [P4].
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_SCALE_F32 = 0,   /* fp32 scales: activation scale = amax / 448 */
    FP8BS_SCALE_UE8M0 = 1, /* e8m0 bytes: activation scale = 2^ceil(log2(amax / 448)) */
} fp8bs_scale_kind;

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_ARG = -1,        /* null pointer, unknown scale kind, bad stride */
    FP8BS_ERR_SHAPE = -2,      /* M, N or K outside the supported range */
    FP8BS_ERR_ALIGN = -3,      /* a pointer or row stride is not 16-byte aligned */
    FP8BS_ERR_SCALE_KIND = -4, /* packed weight holds another scale kind or shape */
    FP8BS_ERR_WORKSPACE = -5,  /* workspace or packed buffer too small / misaligned */
    FP8BS_ERR_CUDA = -6,       /* a CUDA runtime call failed (launch, copy, attribute) */
    FP8BS_ERR_TIMEOUT = -7,    /* device: a bounded wait expired; outputs are invalid */
    FP8BS_ERR_DEVICE = -8,     /* device: another device-side check failed */
    FP8BS_ERR_RESIDENCY = -9,  /* the launch's CTAs cannot all be resident at once; nothing launched */
} fp8bs_status;

/* Largest token count of the fused GEMM.  [P1] "Motivation" fuses up to 32
 * tokens and keeps the library path above; [P2] "Modifications" raises the
 * small-M MoE kernel's cap to 48 tokens at TP8, where the library path slows.
 * Here 33..64 tokens run with a 64-token tile (one CTA per SM). */
#define FP8BS_MAX_M 64

/* Text for a status code.  Never NULL; static storage. */
const char* fp8bs_status_string(int status);

/* Library version, (major << 16) | minor. */
int fp8bs_version(void);

/* ------------------------------------------------------------------------ */
/* Activation quantisation ([P1] "Modifications", the first of the two old   */
/* launches; [P4] "Modifications", ue8m0 per-1x128 quant)                   */
/* ------------------------------------------------------------------------ */

/* Quantise bf16 activations in 1x128 groups along K.
 *   x   : bf16 [M, K], row stride ldx elements.  x and ldx*2 bytes must be
 *         16-byte aligned.
 *   M   : rows, M >= 0 (0 enqueues nothing and returns FP8BS_OK).
 *   K   : multiple of 128, K >= 128.
 *   xq  : e4m3fn codes [M, K], row stride K (8-byte aligned).
 *   xs  : [M, K/128]: fp32 (kind F32, 4-byte aligned) or e8m0 bytes (UE8M0).
 * Per group: amax = max |x| (fp32); F32: s = amax / 448 (IEEE fp32 division);
 * UE8M0: s = smallest power of two >= fp32(amax / 448), exponent clamped to
 * [-127, 127].  Codes = e4m3fn RNE-saturated of x / s (IEEE fp32 division).
 * A group with amax == 0 gets s = 0 (F32) or byte 0 (UE8M0) and signed zeros.
 * Errors: FP8BS_ERR_ARG, FP8BS_ERR_SHAPE, FP8BS_ERR_ALIGN, FP8BS_ERR_CUDA. */
int fp8bs_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int scale_kind,
                uint8_t* xq, void* xs, void* stream);

/* Largest K of fp8bs_rmsnorm_quant (the row stays in registers). */
#define FP8BS_RMSNORM_MAX_K 16384

/* Fused RMSNorm + 1x128 quant: the producer of [P4] "Modifications" (the
 * input_norm / q_norm kernels emit the GEMM's activation scales themselves,
 * so the quant adds no launch).  Its codes and scales feed
 * fp8bs_gemm_prequant.  Per row m, in fp32:
 *   r = 1 / sqrt(sum_k x[m,k]^2 / K + eps)   (IEEE division and square root;
 *                                             r = 0 when the sum and eps are 0)
 *   y[m,k] = bf16_rn((x[m,k] * r) * gamma[k])
 * then y is quantised exactly as fp8bs_quant quantises a bf16 input, so the
 * bytes equal fp8bs_quant applied to the y this call writes.
 *   x     : bf16 [M, K], row stride ldx elements; x and ldx*2 bytes 16-byte
 *           aligned.
 *   M     : rows, M >= 0 (0 enqueues nothing and returns FP8BS_OK).
 *   K     : multiple of 128, 128 <= K <= FP8BS_RMSNORM_MAX_K.
 *   gamma : bf16 [K] RMSNorm weight, 16-byte aligned.
 *   eps   : finite, >= 0.
 *   xq    : e4m3fn codes [M, K], row stride K (8-byte aligned).
 *   xs    : [M, K/128]: fp32 (kind F32, 4-byte aligned) or e8m0 bytes (UE8M0).
 *   y     : optional (NULL to skip) bf16 [M, K] normalised rows, row stride ldy
 *           elements; y and ldy*2 bytes 16-byte aligned.
 * The sum of squares is reduced in a fixed order: repeated calls give the same
 * bytes.  All buffers are the caller's; nothing is allocated or synchronised.
 * Errors: FP8BS_ERR_ARG (kind, eps, null pointer, ldx or ldy < K),
 * FP8BS_ERR_SHAPE, FP8BS_ERR_ALIGN, FP8BS_ERR_CUDA. */
int fp8bs_rmsnorm_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                        const uint16_t* gamma, float eps, int scale_kind, uint8_t* xq,
                        void* xs, uint16_t* y, int64_t ldy, void* stream);

/* Quantise an fp32 weight in 128x128 blocks (the offline producer of the
 * [N/128, K/128] weight scale of [P1] "Modifications"; with UE8M0 each block
 * scale is rounded up to a power of two as in [P4] "Motivation").
 *   w   : fp32 [N, K], row stride ldw elements; w and ldw*4 16-byte aligned.
 *   N,K : multiples of 128, >= 128.
 *   wq  : e4m3fn codes [N, K], row stride K (16-byte aligned).
 *   ws  : [N/128, K/128] fp32 or e8m0 bytes.
 * Same rounding rules as fp8bs_quant, over each 128x128 block. */
int fp8bs_quant_weight(const float* w, int64_t N, int64_t K, int64_t ldw, int scale_kind,
                       uint8_t* wq, void* ws, void* stream);

/* Encode fp32 values to e4m3fn codes with the rounding every kernel of this
 * library uses (round to nearest even, finite magnitudes >= 448 saturate to
 * +-448, NaN in gives NaN out).  A diagnostic of the encoder behind the quant
 * entry points ([P2] "Modifications" names float8_e4m3fn).
 *   v     : fp32 [n], 16-byte aligned.
 *   codes : uint8 [n], 4-byte aligned.
 *   n     : >= 0, a multiple of 4 (0 enqueues nothing). */
int fp8bs_encode_e4m3(const float* v, int64_t n, uint8_t* codes, void* stream);

/* ------------------------------------------------------------------------ */
/* Weight prepack (GB300 layout; replaces the (16,16) pre-shuffle of [P1]    */
/* "Modifications", which is specific to the gfx950 MFMA operand order)     */
/* ------------------------------------------------------------------------ */

/* Bytes of a packed weight: a 256-byte header, N/128 * K/128 tiles of 16384
 * bytes, then the scales (4 or 1 byte per tile), rounded up to 256 bytes.
 * Returns 0 for an invalid shape or kind. */
size_t fp8bs_packed_weight_bytes(int64_t N, int64_t K, int scale_kind);

/* Pack an e4m3fn weight and its block scales for fp8bs_gemm_fused.
 *   wq     : e4m3fn codes [N, K], row stride ldw bytes (wq and ldw 16-byte aligned).
 *   ws     : [N/128, K/128] contiguous: fp32 for F32, e8m0 bytes for UE8M0.
 *   packed : output, >= fp8bs_packed_weight_bytes(N, K, scale_kind) bytes,
 *            256-byte aligned.  Layout: header {magic, version, N, K, kind};
 *            tile (nt, kb) at 256 + (nt * K/128 + kb) * 16384 holding rows
 *            nt*128 .. +127 and columns kb*128 .. +127 of wq in the shared-
 *            memory operand image of a K-major, 128-byte-swizzled MMA tile
 *            (row r, 16-byte chunk j at (r/8)*1024 + (r%8)*128 + ((j^(r%8))*16));
 *            then the scales in [N/128, K/128] order.
 * The packed buffer is read-only for the GEMM and can be shared by any number
 * of concurrent calls.  Errors: ARG, SHAPE, ALIGN, WORKSPACE (too small), CUDA. */
int fp8bs_prepack_weight(const uint8_t* wq, int64_t ldw, const void* ws, int64_t N, int64_t K,
                         int scale_kind, void* packed, size_t packed_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused quant + block-scale GEMM ([P1] "Modifications": one launch per      */
/* linear at M <= 32; here up to FP8BS_MAX_M)                                */
/* ------------------------------------------------------------------------ */

/* Flags of fp8bs_gemm_fused. */
enum {
    /* Launch with programmatic dependent launch: the call may start, and read
     * `packed`, while the kernel before it on the stream is still running; x,
     * y, xq_out, xs_out and the workspace are touched only after that kernel
     * has completed.  Back-to-back linears then overlap one call's start-up
     * and weight stream with the previous call's tail.  Use it only when the
     * work just before this call on the stream does not write `packed`. */
    FP8BS_FLAG_PDL = 1u,
};

/* Workspace bytes the fused GEMM needs for an N x K weight on a device with
 * sm_count multiprocessors (sm_count <= 0: the current device, which needs a
 * CUDA device): a 256-byte error word, 4 KB of epoch words, two 64 KB split-K
 * partial slots per multiprocessor, and 64 x K + 64 x K/128 x 4 bytes for the
 * codes and scales of the two-launch route when the caller does not ask for
 * them.  The size depends on K and sm_count only and every region sits at a
 * place that depends on sm_count only, so a workspace sized for the largest K
 * serves every weight of that K or less.  Returns 0 for an unsupported shape
 * (K/128 must not exceed 10 * sm_count). */
size_t fp8bs_workspace_bytes(int64_t N, int64_t K, int sm_count);

/* Zero a workspace before its first use.  The fused GEMM tags every word it
 * exchanges through the workspace with a per-call epoch kept in the workspace
 * itself, so later calls and graph replays need no re-init.  The epoch is a
 * 32-bit counter that skips 0 (the tag of a word never written since the
 * init) when it wraps, so its period is 2^32 - 1 calls.  A stale word is
 * taken for current only if it was last written a whole number of periods
 * before and not since: calls of one shape rewrite every word they read, so
 * that needs a word left idle (a larger M or another split of the same
 * workspace) for exactly that many calls; a re-init before reusing a
 * workspace across such spans rules it out. */
int fp8bs_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Y = bf16(x W^T) with the 1x128 activation quant fused in.
 *   x        : bf16 [M, K], row stride ldx; x and ldx*2 16-byte aligned.
 *   M        : 1 .. FP8BS_MAX_M (0 enqueues nothing and returns FP8BS_OK).
 *   N, K     : multiples of 128 with K/128 <= 10 * (multiprocessor count).
 *              Weights with more than 10 * (multiprocessor count) 128x128
 *              tiles are processed in several launches of whole 128-row
 *              slices.
 *   packed   : from fp8bs_prepack_weight with the same N, K and scale_kind;
 *              packed_bytes its size (checked against N, K, kind on the host;
 *              the header is checked on the device).
 *   y        : bf16 [M, N], row stride ldy >= N (y and ldy*2 16-byte aligned).
 *   workspace: >= fp8bs_workspace_bytes(N, K, 0) bytes, 256-byte aligned,
 *              initialised once by fp8bs_workspace_init.  One workspace must not
 *              be used by two calls that can run at the same time.
 *   xq_out, xs_out : optional (NULL to skip) copies of the quantised
 *              activations ([M, K] codes, row stride K; [M, K/128] scales),
 *              bit-identical to fp8bs_quant.
 *   flags    : 0 or FP8BS_FLAG_PDL.
 * The result is deterministic: the split-K partials are summed in a fixed
 * order, so repeated calls and graph replays give identical bits.
 * Up to 32 tokens the call is one launch (measured faster than the pair
 * below at every such token count).  From 33 tokens on it is two: the 1x128
 * quant (into xq_out / xs_out when given, else into the workspace), then the
 * GEMM on those codes, the same kernels as fp8bs_quant followed by
 * fp8bs_gemm_prequant and bit-identical to them (with FP8BS_FLAG_PDL both
 * launch with programmatic dependent launch).
 * The CTAs of one launch exchange data, so a call assumes the whole device:
 * one CTA per multiprocessor, all resident together.  Before each launch the
 * library checks that the kernel's occupancy (CTAs per multiprocessor at its
 * shared memory and thread count) times the device's multiprocessors covers
 * the grid, and returns FP8BS_ERR_RESIDENCY without launching if not.  It
 * cannot see kernels of other streams or processes that hold
 * multiprocessors: there the bounded waits expire and the call reports
 * FP8BS_ERR_TIMEOUT.
 * Errors (host): ARG, SHAPE, ALIGN, WORKSPACE, CUDA, RESIDENCY.  Errors
 * (device, via fp8bs_check_error): SCALE_KIND (header mismatch; y not
 * written), TIMEOUT. */
int fp8bs_gemm_fused(const uint16_t* x, int64_t M, int64_t ldx, const void* packed,
                     size_t packed_bytes, int64_t N, int64_t K, int scale_kind, uint16_t* y,
                     int64_t ldy, void* workspace, size_t workspace_bytes, uint8_t* xq_out,
                     void* xs_out, unsigned flags, void* stream);

/* The GEMM on activations quantised beforehand: the second launch of the
 * two-launch path ([P1] "Motivation": the per-1x128 quant and the block-scale
 * GEMM as separate kernels, the path the fused call replaces; "Kernel
 * microbenchmarks" times the two against it).  fp8bs_quant followed by this
 * call gives a Y bit-identical to fp8bs_gemm_fused on the same x: the MMAs,
 * the rescale and the split-K order are the same.
 *   xq   : e4m3fn codes [M, K], row stride ldxq (xq and ldxq 16-byte aligned).
 *   xs   : [M, K/128] scales, fp32 (4-byte aligned) or e8m0 bytes, of the
 *          kind scale_kind (the packed weight's kind).
 * Everything else as fp8bs_gemm_fused (flags: 0 or FP8BS_FLAG_PDL).
 * Errors (host): ARG, SHAPE, ALIGN, WORKSPACE, CUDA.  Errors (device, via
 * fp8bs_check_error): SCALE_KIND, TIMEOUT. */
int fp8bs_gemm_prequant(const uint8_t* xq, int64_t M, int64_t ldxq, const void* xs, const void* packed,
                        size_t packed_bytes, int64_t N, int64_t K, int scale_kind, uint16_t* y,
                        int64_t ldy, void* workspace, size_t workspace_bytes, unsigned flags,
                        void* stream);

/* Synchronise `stream`, read the workspace error word, clear it, and return
 * FP8BS_OK or the first device-side status recorded since the last check.
 * After FP8BS_ERR_TIMEOUT the epoch words may disagree: call
 * fp8bs_workspace_init before the workspace is used again. */
int fp8bs_check_error(void* workspace, void* stream);

/* ------------------------------------------------------------------------ */
/* Small-M FP8 block-scale MoE layer ([P2] "Modifications")                  */
/* ------------------------------------------------------------------------ */

#define FP8BS_MOE_MAX_PAIRS 1024    /* M * S: routed (token, slot) pairs    */
#define FP8BS_MOE_MAX_EXPERTS 4096  /* E                                     */
#define FP8BS_MOE_MAX_I 512         /* intermediate size per expert          */

/* Workspace bytes of fp8bs_moe_w8a16: a 256-byte error word, the gate/up
 * partial sums (M*S x H/512 x 2I fp32) and the per-slot down projections
 * (M*S x H fp32).  Returns 0 for an unsupported shape. */
size_t fp8bs_moe_workspace_bytes(int64_t M, int64_t S, int64_t H, int64_t I);

/* One MoE layer at decode sizes, the FP8 small-M kernel of [P2]
 * "Modifications": float8_e4m3fn w13 / w2 with contiguous 128x128 fp32 block
 * scales, each block's scale applied to its partial sum, bf16 activations,
 * routing given per token (no sort).  Per token m and slot s, with
 * e = topk_ids[m, s]:
 *   h    = x[m] . w13[e]^T   (w13[e] stacks the gate rows 0..I-1 over the up
 *                             rows I..2I-1; per 128-wide K block the partial
 *                             sum times its scale, fp32)
 *   a    = bf16(silu(h_gate) * h_up),  silu(g) = g / (1 + exp(-g))
 *   o    = a . w2[e]^T        (same block-scale rule)
 *   y[m] = bf16(sum over s, in slot order, of topk_w[m, s] * o)
 *   x        : bf16 [M, H], 16-byte aligned, rows contiguous; finite values
 *              below 2^64 in magnitude (the weights are decoded as exact
 *              power-of-two-scaled values, and x carries the 2^64).
 *   M, S     : tokens and slots per token, M >= 0 (0 is a no-op), S >= 1,
 *              M * S <= FP8BS_MOE_MAX_PAIRS.
 *   H        : hidden size, a multiple of 512.
 *   topk_ids : int32 [M, S] expert ids; an id outside [0, E) makes that slot
 *              contribute nothing and records FP8BS_ERR_DEVICE in the
 *              workspace error word.
 *   topk_w   : fp32 [M, S] routing weights.
 *   w13, s13 : e4m3fn [E, 2I, H] (16-byte aligned), fp32 [E, 2I/128, H/128].
 *   w2, s2   : e4m3fn [E, H, I] (16-byte aligned), fp32 [E, H/128, I/128].
 *   E, I     : experts (1..FP8BS_MOE_MAX_EXPERTS); I in {128, 256, 512}.
 *   y        : bf16 [M, H], 8-byte aligned.
 *   workspace: fp8bs_moe_workspace_bytes(M, S, H, I) bytes, 256-byte aligned;
 *              its first word must be zero before the first call (e.g.
 *              fp8bs_workspace_init); fp8bs_check_error reads it.
 * Three launches on `stream` (gate/up, down, combine), the last two with
 * programmatic dependent launch; no cross-CTA waits; every sum in a fixed
 * order, so results are deterministic.  Each active expert's weights are read
 * once per call, whatever number of tokens it serves.
 * Errors: FP8BS_ERR_SHAPE, FP8BS_ERR_ARG, FP8BS_ERR_ALIGN,
 * FP8BS_ERR_WORKSPACE, FP8BS_ERR_CUDA. */
int fp8bs_moe_w8a16(const uint16_t* x, int64_t M, int64_t H, const int32_t* topk_ids,
                    const float* topk_w, int64_t S, const uint8_t* w13, const float* s13,
                    const uint8_t* w2, const float* s2, int64_t E, int64_t I, uint16_t* y,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Limits of fp8bs_gemm_fused_static's fixed scratch. */
#define FP8BS_STATIC_MAX_K 16384  /* largest K it accepts                   */
#define FP8BS_STATIC_MAX_SMS 160  /* CTAs it uses at most (grid cap)        */

/* fp8bs_gemm_fused without a workspace argument: the scratch lives in one
 * fixed device array inside this library (22,057,216 bytes per device,
 * sized for FP8BS_STATIC_MAX_SMS CTAs and K up to FP8BS_STATIC_MAX_K), so the
 * call allocates no device memory, ever.  It is meant for callers that cannot
 * allocate or own device memory: an operator plugged into a runtime whose
 * device memory is handed out up front to its own pool (a serving engine that
 * reserves all free HBM for its KV cache), a callback that gets no allocator
 * handle, or a latency-critical path where an allocation's implicit device
 * synchronisation is not acceptable.  The pages describe no counterpart: it is
 * a deployment convenience around the same kernel.
 *
 * Arguments, results and host checks are those of fp8bs_gemm_fused, except:
 *   K > FP8BS_STATIC_MAX_K is refused with FP8BS_ERR_WORKSPACE (the scratch
 *   is too small); on a device with more than FP8BS_STATIC_MAX_SMS
 *   multiprocessors the call uses that many CTAs.
 *   status_out: optional (NULL to skip) device uint32 that receives, in stream
 *   order after the kernel, the scratch's error word: 0, or the negated
 *   status (FP8BS_ERR_TIMEOUT, FP8BS_ERR_SCALE_KIND) of the first device-side
 *   failure since the last call that passed a status_out; the word is then
 *   cleared in stream order.  After a timeout the scratch's epoch words may
 *   disagree, and this entry point cannot re-initialise them: later calls may
 *   time out too.
 * Set-up: the first call on each device (with that device current) looks up
 * the array's address with cudaGetSymbolAddress, zeroes it on `stream` and
 * waits for that.  Make that first call outside stream capture: on a
 * capturing stream it returns FP8BS_ERR_ARG and enqueues nothing.
 * Sharing: every call on one device uses the same array, so two calls that
 * can overlap (different streams, different host threads without ordering)
 * race and may time out or return wrong results.  Calls in order on one
 * stream, with or without FP8BS_FLAG_PDL, are safe. */
int fp8bs_gemm_fused_static(const uint16_t* x, int64_t M, int64_t ldx, const void* packed,
                            size_t packed_bytes, int64_t N, int64_t K, int scale_kind,
                            uint16_t* y, int64_t ldy, uint8_t* xq_out, void* xs_out,
                            uint32_t* status_out, unsigned flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Timeline tracing (profiling aid; no counterpart on the pages)             */
/* ------------------------------------------------------------------------ */

#define FP8BS_TRACE_CALLS 256  /* calls kept, by workspace epoch modulo 256  */
#define FP8BS_TRACE_CTAS 160   /* CTAs kept per call                         */
#define FP8BS_TRACE_POINTS 64  /* phase stamps per CTA                       */

/* Copy the per-phase timeline of the fused GEMM's most recent calls to host
 * memory.  Only a library built with tracing records one (native_build's
 * trace=True, which compiles the kernels with FP8BS_TRACE; every CTA then
 * stamps its phase boundaries with %globaltimer and clock64); the plain
 * library keeps no timeline, returns FP8BS_ERR_ARG and copies nothing.
 *   host_dst: host buffer of `bytes` bytes; receives the first `bytes` bytes of
 *             uint64 [FP8BS_TRACE_CALLS][FP8BS_TRACE_CTAS][FP8BS_TRACE_POINTS][2]
 *             (globaltimer ns, clock64 cycles), call slot = the call's
 *             workspace epoch modulo FP8BS_TRACE_CALLS, point order as in the
 *             library's csrc/trace.cuh; a stamp that was not taken is 0.
 * Synchronises with the device (a blocking copy).  Errors: FP8BS_ERR_ARG (no
 * tracing in this build, or a null buffer), FP8BS_ERR_CUDA. */
int fp8bs_trace_read(void* host_dst, size_t bytes);

/* ------------------------------------------------------------------------ */
/* Diagnostic settings (for the library's own tests; no counterpart on the  */
/* pages)                                                                    */
/* ------------------------------------------------------------------------ */

/* Override, for the calls that follow in this process, two settings of the
 * fused GEMM's launches:
 *   timeout_cycles   : the limit of every bounded wait inside the kernel, in
 *                      SM clock cycles; <= 0 restores the default (2e9,
 *                      about 1 s), which is set far above any legitimate wait.
 *                      A short limit (1e5 .. 1e6) makes a wait that cannot
 *                      complete expire quickly, so a test can drive the
 *                      expiry path (FP8BS_ERR_TIMEOUT, drain, return).
 *   sm_count_override: the multiprocessor count the library sizes grids and
 *                      workspaces for; <= 0 restores the device's own.  The
 *                      residency check still uses the device's real count, so
 *                      a large override makes a call return
 *                      FP8BS_ERR_RESIDENCY without launching.
 * Process-wide, not synchronised with calls in flight on other host threads.
 * Returns FP8BS_OK. */
int fp8bs_debug_config(long long timeout_cycles, int sm_count_override);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
