/*
 * skinny.h -- C ABI of libskinny, the weight-only "skinny" linear layer for
 * GB300 (sm_103a):
 *
 *     y[m][n] = sum_k x[m][k] * w[n][k]      m < M <= 8,  n < N,  k < K
 *
 * with FP16 activations x and weights w that stay compressed in device memory
 * and are decoded in registers inside the kernel, with no "dequantize the
 * model first" pass.  This is the decode-time linear layer of the pages'
 * system: weight bandwidth dominates single-request decode, the weights are
 * read compressed from HBM and each small piece is turned into FP16 register
 * operands (page "NVFP4 在 Volta 上！", section "我实际构建了什么"); M = 1 is one
 * decode token, M = 8 the k=7 speculative-verify round packed as 8 rows (same
 * page, kernel table "路径 有效带宽 测量读取上限" and the paragraph after it).
 *
 * Weight formats (the pages name NVFP4 and FP8-E4M3 regions of the checkpoint,
 * page "NVFP4 在 Volta 上！", section on v1.1; the layouts are this library's):
 *
 *   NVFP4  W_codes  u8 [N][K/2]  two E2M1 codes per byte, LOW nibble = even k
 *          W_scales u8 [N][K/16] one E4M3 scale per 16 consecutive k of a row
 *          W_gscale f32          one tensor scale
 *          w[n][k] = E2M1(code) * E4M3(W_scales[n][k/16]) * W_gscale
 *   FP8    W_codes  u8 [N][K]    E4M3 codes
 *          W_scales f32 [ceil(N/128)][ceil(K/128)] one scale per 128x128 block
 *          w[n][k] = E4M3(code) * W_scales[n/128][k/128]
 *
 *   E2M1 is the OCP MX FP4 element type; E4M3 is the OCP OFP8 "E4M3" type
 *   (no infinities, S.1111.111 = NaN).
 *
 * Common rules for every entry point
 *   - x is FP16, row-major [M][K]; y is row-major [M][N].  All pointers are
 *     device pointers owned by the caller; the library keeps none of them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream), do no host synchronisation and allocate nothing: the
 *     split-K partial sums and the argmax partials live in the workspace that
 *     sk_init() allocated for the current device.
 *   - Arguments are checked before anything is launched; a rejected call
 *     launches nothing and returns the status code.  Launch failures return
 *     SK_ERR_CUDA.
 *   - Determinism: a given (shape, device) always sums in the same order, so
 *     repeated calls are bitwise identical.  Split-K partials are combined in a
 *     fixed order, never with floating-point atomics.
 *   - Accuracy contract (FP32 accumulation of exact FP16 products):
 *       |y - y_exact| <= 1e-3 * sum_k |x[m][k] * w[n][k]| + 1e-6
 *     plus one FP16 ulp of the result for the *_f16out variants.
 *   - One stream at a time per workspace: calls whose kernels overlap in time
 *     on different streams of the same device race on the workspace.  Each
 *     kernel also expects its whole grid (two CTAs per SM) to be resident at
 *     once -- its split-K owners wait for partial sums from the other CTAs of
 *     the grid -- so
 *     another kernel that occupies SMs at the same time can make those waits
 *     run out (SK_ERR_TIMEOUT) instead of finishing.  Streams that must run
 *     at the same time each get a workspace of their own with
 *     sk_stream_workspace(); their calls then launch cooperatively (the whole
 *     grid resident before it starts), which rules both problems out.
 *     Consecutive calls on one stream may overlap through programmatic
 *     dependent launch (PDL): a linear kernel may start streaming its own
 *     weights while the kernel before it on the stream finishes, but touches
 *     x, y and the workspace only after that kernel has completed.  Weights
 *     are therefore read before the preceding kernel is known to be done:
 *       * the library's own weight writers, fp8_quantize and nvfp4_quantize,
 *         mark their stream, and the next linear call on that stream is
 *         launched without PDL, so quantize-then-multiply on one stream is
 *         safe with no synchronisation in between;
 *       * a kernel from outside the library that writes the weights must not
 *         be the kernel immediately preceding a linear call on the same
 *         stream while PDL is on (sk_set_pdl(0) turns it off); anything
 *         launched in between without PDL -- any other kernel, a copy, an
 *         event wait -- ends the hazard.
 *   - Kernels bound every wait they spin on (about one second).  When a wait
 *     runs out the kernel records SK_ERR_TIMEOUT in a device word, finishes
 *     without further waiting and leaves garbage in y; sk_last_device_error()
 *     reports it, and the workspace must then be re-created with sk_init().
 */
#ifndef SKINNY_H
#define SKINNY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SK_API __attribute__((visibility("default")))
#else
#define SK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SK_OK = 0,
    SK_ERR_INVALID_ARG = 1,       /* NULL pointer, M outside 1..8, negative N/K */
    SK_ERR_UNSUPPORTED_SHAPE = 2, /* K not a multiple of 256 (NVFP4) / 128 (FP8) */
    SK_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rule of its argument */
    SK_ERR_NOT_INITIALIZED = 4,   /* no sk_init() on the current device */
    SK_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
    SK_ERR_TIMEOUT = 6,           /* a bounded in-kernel wait ran out (sk_last_device_error) */
    SK_ERR_WORKSPACE = 7          /* the workspace is too small for this call's partial sums */
} sk_status;

/*
 * Allocate (cudaMalloc) and initialise the workspace of the CURRENT device
 * (a zeroed 4 KiB control block followed by split-K partial-sum slots, all
 * marked empty; every call leaves them empty again).
 * workspace_bytes = 0 picks the default, 64 MiB, which covers the largest call
 * below (N = 151936, K = 5120, M = 8 needs about 25 MB).  Calling it again on
 * the same device frees and re-creates the workspace (wait for all work of the
 * library on that device first).  Call it before capturing any CUDA graph.
 * It also resolves cuTensorMapEncodeTiled from the driver.
 */
SK_API sk_status sk_init(size_t workspace_bytes);

/*
 * A workspace of its own for `stream` (a cudaStream_t; NULL = the legacy
 * default stream) on the CURRENT device, allocated (cudaMalloc) and initialised
 * like sk_init's; workspace_bytes = 0 removes the stream's workspace (its calls
 * fall back to the device's).  Calling it again replaces the workspace (after
 * synchronising the stream).  Every later call on that stream -- linear
 * layers, lm_head, quantizers, sk_last_device_error -- uses it instead of the
 * device's, and its linear-layer kernels are launched cooperatively, so that
 * the whole persistent grid is resident before any of its CTAs starts: calls
 * on streams that each have a workspace of their own can then overlap on the
 * GPU without racing on a workspace and without a split-K wait that could run
 * out.  A cooperative kernel starts only when the whole grid fits, so
 * overlapping calls share the SMs in turns rather than at once; such calls
 * are also launched without programmatic dependent launch.  Up to 64 stream
 * workspaces per process; more return SK_ERR_INVALID_ARG.  Call it before
 * capturing a CUDA graph.  Needs no sk_init() (the device's workspace is
 * only the fallback).
 */
SK_API sk_status sk_stream_workspace(void *stream, size_t workspace_bytes);

/* Free the workspaces of all devices and streams (synchronises each device first). */
SK_API sk_status sk_shutdown(void);

/*
 * NVFP4 weight-only linear, FP32 output y[M][N].
 *   x        const f16 [M][K], 16-byte aligned (32-byte aligned x is read with
 *            wider loads from M = 4 on, a little faster; the results are the same)
 *   W_codes  const u8 [N][K/2], 16-byte aligned
 *   W_scales const u8 [N][K/16], 16-byte aligned
 *   W_gscale FP32 tensor scale (any finite value)
 *   y        f32 [M][N], 4-byte aligned
 *   1 <= M <= 8; N >= 0 (N = 0: nothing is launched); K >= 0 with
 *   K % 256 == 0 (K = 0: y is set to zero).
 */
SK_API sk_status nvfp4_gemm(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                     float W_gscale, float *y, int M, int N, int K, void *stream);

/* As nvfp4_gemm, FP16 output (round to nearest even), y 2-byte aligned. */
SK_API sk_status nvfp4_gemm_f16out(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                            float W_gscale, void *y, int M, int N, int K, void *stream);

/*
 * FP8-E4M3 weight-only linear with FP32 128x128 block scales, FP32 output.
 *   x        const f16 [M][K], 16-byte aligned (32-byte: as nvfp4_gemm)
 *   W_codes  const u8 [N][K], 16-byte aligned
 *   W_scales const f32 [ceil(N/128)][ceil(K/128)], 4-byte aligned
 *   y        f32 [M][N], 4-byte aligned
 *   1 <= M <= 8; N >= 0; K >= 0 with K % 128 == 0.
 */
SK_API sk_status fp8_gemm(const void *x, const uint8_t *W_codes, const float *W_scales,
                   float *y, int M, int N, int K, void *stream);

/* As fp8_gemm, FP16 output, y 2-byte aligned. */
SK_API sk_status fp8_gemm_f16out(const void *x, const uint8_t *W_codes, const float *W_scales,
                          void *y, int M, int N, int K, void *stream);

/*
 * NVFP4 vocabulary projection with a fused greedy pick: the logits are those
 * of nvfp4_gemm and argmax[m] is the lowest n holding the maximum of row m of
 * those same FP32 logits (the greedy / local-argmax proposal that the
 * speculative verify round compares against, page "NVFP4 在 Volta 上！",
 * section "这是一个服务器，不是 GEMM 截图"; native 4-bit lm_head, kernel table).
 *   logits  f32 [M][N] or NULL (then only argmax is written)
 *   argmax  i32 [M], 4-byte aligned
 *   Other arguments as nvfp4_gemm; N >= 1.  NaN logits (not produced by
 *   finite inputs) would order above +inf.
 */
SK_API sk_status lm_head_argmax(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                         float W_gscale, float *logits, int32_t *argmax,
                         int M, int N, int K, void *stream);

/*
 * lm_head_argmax plus the greedy verification of one speculative round, in the
 * same kernel's final step (page "NVFP4 在 Volta 上！": the k = 7 MTP round is
 * verified on eight rows, and each round commits a prefix of the drafts plus
 * one token of the target's own).  Row m of x is the target's state after the
 * prefix and the first m drafted tokens, so argmax[m] is the target's pick for
 * the position that draft[m] proposes.
 *   draft   const i32 [M - 1]: the drafted tokens (may be NULL when M == 1),
 *           4-byte aligned, device memory
 *   accept  i32 [2], 4-byte aligned: accept[0] = a, the number of leading
 *           drafts with draft[j] == argmax[j] for every j < a; accept[1] =
 *           argmax[a], the token the target commits after them (a + 1 tokens
 *           are committed in all)
 *   Other arguments as lm_head_argmax.  K = 0 is rejected with
 *   SK_ERR_UNSUPPORTED_SHAPE (no logits to verify against).
 */
SK_API sk_status lm_head_verify(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                                float W_gscale, float *logits, int32_t *argmax, const int32_t *draft,
                                int32_t *accept, int M, int N, int K, void *stream);

/*
 * Weight quantizers: FP16 -> the formats above, on the GPU (the conversion step
 * before the linear layers; the pages convert an FP16 checkpoint to NVFP4 --
 * v100-skinny ai-manual.ru article, section "Конвертация модели в NVFP4" -- and
 * keep FP8 regions in FP8, page "NVFP4 在 Volta 上！", v1.1 section -- but
 * print no rounding rules, so this library fixes them).  Every step is an IEEE
 * binary32 operation rounded to nearest-even, in the order given; the final
 * roundings are nearest-even, ties to the even mantissa, saturating at the
 * format's maximum, keeping the input's sign (also for zero).  Results are
 * therefore bit-for-bit reproducible.  w is FP16 row-major [N][K], 16-byte
 * aligned, device memory, with finite values (infinities or NaNs give
 * unspecified codes); outputs are device memory owned by the caller.
 *
 * fp8_quantize, per 128 x 128 block (the last row / column of blocks may be
 * partial):  a = max |w| over the block;  s = a / 448 (s = 1 when a = 0);
 * code = E4M3(w / s).
 *   codes  u8 [N][K], 8-byte aligned;  scales f32 [ceil(N/128)][ceil(K/128)]
 *   K % 8 == 0 (fp8_gemm itself needs K % 128 == 0).  N or K = 0: no-op.
 */
SK_API sk_status fp8_quantize(const void *w, uint8_t *codes, float *scales, int N, int K, void *stream);

/*
 * nvfp4_quantize, two-level scale:  A = max |w| over the tensor;
 * G = A / 2688 (2688 = 448 * 6; G = 1 when A = 0), written to *gscale; per row
 * and 16 consecutive k:  b = max |w| over them;  sc = E4M3((b / 6) / G);
 * S = the value of sc;  code = E2M1(w / (S * G)) (S = 0: signed zeros).
 *   codes  u8 [N][K/2] (low nibble = even k), 8-byte aligned
 *   scales u8 [N][K/16];  gscale f32 [1], 4-byte aligned, device memory
 *   K % 16 == 0 (nvfp4_gemm itself needs K % 256 == 0).  Needs sk_init() on
 *   the current device (the tensor maximum is gathered in its workspace), and
 *   the workspace's one-stream-at-a-time rule applies.
 */
SK_API sk_status nvfp4_quantize(const void *w, uint8_t *codes, uint8_t *scales, float *gscale, int N, int K,
                                void *stream);

/*
 * NVFP4 vocabulary projection with a sampled pick per row: temperature, top-k
 * and top-p, with the random draw passed in (the pages' server samples at a
 * temperature besides the greedy pick -- page "NVFP4 在 Volta 上！", the
 * "温度 0.6" run -- but gives no sampler, so this library fixes the usual
 * rule).  For row m of the FP32 logits z (those of nvfp4_gemm):
 *   1. candidates: the top_k largest z, ordered by z descending, ties by the
 *      lower index;
 *   2. p_j = exp((z_j - z_0) / temperature) over them (z_0 the largest);
 *   3. keep the shortest prefix whose running sum of p reaches top_p times
 *      the sum over all candidates (at least one candidate);
 *   4. token[m] = the first kept candidate whose running sum exceeds u[m]
 *      times the sum over the kept prefix.
 *   temperature <= 0 gives the greedy pick (the first candidate).  Sums are
 *   FP32 in a fixed order, so a call is reproducible; where u[m] lands within
 *   FP32 rounding of a boundary, an exact-arithmetic sampler may pick the
 *   neighbouring candidate.
 *   logits  f32 [M][N] (written; needed as scratch), 4-byte aligned
 *   u       const f32 [M], uniforms in [0, 1), device memory, 4-byte aligned
 *   token   i32 [M], 4-byte aligned
 *   1 <= top_k <= min(N, 1024) (larger: SK_ERR_UNSUPPORTED_SHAPE);
 *   0 < top_p <= 1; other arguments as nvfp4_gemm with N, K >= 1.
 */
SK_API sk_status lm_head_sample(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                                float W_gscale, float *logits, const float *u, float temperature, int top_k,
                                float top_p, int32_t *token, int M, int N, int K, void *stream);

/* Static, human-readable name of a status code. */
SK_API const char *sk_status_string(sk_status status);

/*
 * Wait for `stream`, then read and clear the device error word of the
 * workspace that calls on `stream` use (the stream's own, else the current
 * device's): SK_ERR_TIMEOUT if a kernel's bounded wait ran out since the last
 * call, SK_OK otherwise (SK_ERR_CUDA if the synchronisation itself failed).
 */
SK_API sk_status sk_last_device_error(void *stream);

/*
 * Programmatic dependent launch between consecutive calls on one stream:
 * 1 = on (default), 0 = off.  Process-wide; returns the previous setting.
 */
SK_API int sk_set_pdl(int enable);

/*
 * Kernel variant, process-wide; returns the previous setting, or -1 (and
 * changes nothing) for a value outside the three below.
 *   SK_VARIANT_AUTO (default): the tensor-core variant (swap-AB m16n8k16 MMA,
 *     tokens padded to 8) for every M, except M = 1 on shapes with many work
 *     units (16 rows x 1024 k) per CTA -- at least 24 for FP8, 96 for NVFP4 --
 *     where the single-token SIMT variant (mixed FP16 x FP16 + FP32 FMA) is
 *     faster.  Both thresholds are measured on GB300.
 *   SK_VARIANT_TENSOR: the tensor-core variant for every M.
 *   SK_VARIANT_SIMT: the SIMT variant for M = 1 (tensor-core for M > 1).
 * Both variants meet the same accuracy bound; each is bitwise reproducible,
 * but they sum in different orders, so their results differ in the last bits.
 */
enum { SK_VARIANT_AUTO = 0, SK_VARIANT_TENSOR = 1, SK_VARIANT_SIMT = 2 };
SK_API int sk_set_variant(int variant);

/*
 * Failure-injection hook for tests: with enable = 1 the next kernel launched
 * by this process on any device issues no weight copies, so its consumers'
 * bounded waits run out (about one second); the kernel then finishes without
 * further waiting and records SK_ERR_TIMEOUT, which sk_last_device_error()
 * returns.  The hook clears itself after that one launch.  No fault, trap or
 * unbounded wait is involved.
 */
SK_API void sk_inject_wait_timeout(int enable);

/*
 * nvfp4_gemm for callers that cannot allocate device memory (the pages have no
 * counterpart; this is a library service).  nvfp4_gemm needs the workspace
 * that sk_init() gets with cudaMalloc; code that must not allocate (inside an
 * arena or pool allocator that owns all device memory, behind an allocator
 * frozen after start-up, on a serving path with a no-allocation rule) calls
 * this instead.  Its scratch memory is a fixed 8 MiB static device array,
 * created when the library is loaded and held by every GPU that loads it until
 * the process exits; the call itself allocates nothing (no cudaMalloc or
 * cudaFree, no library allocation) and needs no sk_init().
 *   Arguments, layouts and results are those of nvfp4_gemm (FP32 output).
 *   SK_ERR_WORKSPACE: the split-K partial sums of this shape do not fit the
 *   array.  With K > 1024 a call needs
 *       ceil(N/16) * ceil(K/1024) * 64 * m  bytes  <=  8,384,512 bytes,
 *   where m is the token slots of the kernel variant that runs: m = 8 for
 *   every M >= 2, and for M = 1 unless the single-token variant is chosen
 *   (sk_set_variant(SK_VARIANT_SIMT), or SK_VARIANT_AUTO on a shape with at
 *   least 96 units of 16 rows x 1024 k per CTA), where m = 1.  For example
 *   at M = 2 and K = 5120, N <= 52,400 fits and N = 52,416 is rejected.
 *   K <= 1024 needs no partial sums.
 *   The first call on a device (with that device current) looks up the
 *   array's device address (cudaGetSymbolAddress), the tensor-map encoder and
 *   the SM count: make it before any stream capture.  All calls share the one
 *   array; each call resets the control block and marks the partial-sum slots
 *   it needs empty before its kernel runs (one small fill kernel).  Calls
 *   whose kernels overlap on the GPU (different streams or host threads) race
 *   on the array.  Bounded-wait timeouts of this entry point are not reported
 *   by sk_last_device_error(); the next call starts from a reset control block
 *   and empty slots, so it is correct again.
 */
SK_API sk_status nvfp4_gemm_noalloc(const void *x, const uint8_t *W_codes, const uint8_t *W_scales,
                                    float W_gscale, float *y, int M, int N, int K, void *stream);

/* Library version, major * 10000 + minor * 100 + patch. */
SK_API int sk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_H */
