/*
 * qswiglu.h -- C ABI of libqswiglu.so, the GB300 (sm_103a) fused
 * weight-quantised SwiGLU expansion
 *
 *     hidden = silu(x . Wg^T) * (x . Wu^T)
 *
 * Source of the operation: mlx-bun source-diff pages ("mlx-bun 0.0.7 -> 0.0.9,
 * page 42" and "mlx-bun 0.0.8 -> 0.0.10, page 41"), file
 * src/model/fused-swiglu-kernel.ts: the header comment (what is fused, the MATCH
 * and F32 precision variants, down_proj left as a separate quantised matmul),
 * fusedSwigluSupported() (accepted quantisation specs) and fusedSwiglu()
 * (shapes, "caller owns" the result).  The standalone quantised linear follows
 * src/model/steel-linear-kernel.ts, steelLinear(), on page 43 ("mlx-bun 0.0.7 ->
 * 0.0.9, page 43").
 *
 * Data layout (all row-major, contiguous, device memory unless stated):
 *   x        bf16  [M, H]                 activation
 *   w        uint32 [rows, H*bits/32]     packed codes; code k of a row sits at
 *                                         bits (k mod pf)*bits of word k/pf,
 *                                         pf = 32/bits (little-endian, LSB first)
 *   scales   bf16  [rows, H/gs]           one scale per group of gs consecutive k
 *   biases   bf16  [rows, H/gs]           affine offsets ("zero points")
 *   dequantised weight  w[r,k] = bf16_rne(scale[r,k/gs] * q[r,k] + bias[r,k/gs])
 *   hidden   bf16  [M, I]
 *
 * Ownership: the caller allocates and owns every buffer; the library keeps no
 * pointer after a call returns and allocates no device memory.
 *
 * Execution: every entry point that takes `stream` (a cudaStream_t passed as
 * void*, NULL = the legacy default stream) only enqueues work on that stream
 * and returns; results are ready when the stream is synchronised.  The calling
 * thread's current CUDA device must be the one that owns the buffers.
 *
 * Errors: argument errors are detected on the host before anything is launched
 * (QSW_ERR_INVALID_ARG / QSW_ERR_UNSUPPORTED, nothing enqueued).  A failed
 * launch returns QSW_ERR_CUDA.  Kernels never trap: a device-side wait that
 * runs past its limit sets a device error word and the kernel exits; the word
 * is read (and cleared) by qsw_check_device_errors().  Nothing is thrown across
 * the ABI.
 */
#ifndef QSWIGLU_H_
#define QSWIGLU_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QSW_API __attribute__((visibility("default")))
#else
#define QSW_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSW_OK = 0,
    QSW_ERR_INVALID_ARG = 1,   /* null pointer, negative size, shape inconsistency */
    QSW_ERR_UNSUPPORTED = 2,   /* valid but not handled: bits, gs, H, alignment, size */
    QSW_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed */
    QSW_ERR_TIMEOUT = 4,       /* a kernel gave up on a device-side wait */
    QSW_ERR_BOUNDS = 5         /* debug build only: a device-side address or copy check failed */
} qsw_status;

/* Rounding variants of the fused expansion (fused-swiglu-kernel.ts, header
 * comment "PRECISION"; debug variants mirror its SWIGLU_DEBUG_GATE switch). */
typedef enum {
    QSW_MATCH = 0,       /* gate,up -> bf16; sigma, silu, product each rounded to bf16 */
    QSW_F32 = 1,         /* gate, up, sigma, silu kept f32; one rounding at the store */
    QSW_DEBUG_GATE = 2,  /* hidden := bf16(x . Wg^T), the stored gate projection */
    QSW_DEBUG_UP = 3     /* hidden := bf16(x . Wu^T), the stored up projection */
} qsw_variant;

/* Activation dtype of the *_ex entry points: x, the scales and biases of
 * both operands, and the result (fusedSwigluSupported() accepts bf16 or f16
 * activations; the dequantised weights, the stored projections and every MATCH
 * rounding are in the same dtype).  The other entry points are bf16. */
typedef enum {
    QSW_ACT_BF16 = 0,
    QSW_ACT_F16 = 1
} qsw_act_dtype;

/* Indices into the dispatch counters (fused-swiglu-kernel.ts keeps a call
 * counter so a test can prove the kernel ran). */
enum {
    QSW_CNT_FUSED_TC = 0,     /* fused expansion, tensor-core (tcgen05) kernel */
    QSW_CNT_FUSED_GEMV = 1,   /* fused expansion, small-M kernel */
    QSW_CNT_QMM_TC = 2,       /* affine_qmm, tensor-core kernel */
    QSW_CNT_QMM_GEMV = 3,     /* affine_qmm, small-M kernel */
    QSW_CNT_SILU_MUL = 4,     /* elementwise silu*mul */
    QSW_CNT_GEMV_STREAM = 5,  /* small-M calls (fused or affine_qmm) served by the warp-streamed kernel */
    QSW_NUM_COUNTERS = 6
};

/*
 * Fused expansion hidden[M,I] = epilogue(x . Wg^T, x . Wu^T).
 * Gate and up carry their own (gs, bits): fusedSwigluSupported() allows mixed
 * specs.  Accepted: M >= 0 (M = 0 enqueues nothing), H >= 32, I >= 1,
 * bits in {2,4,8}, gs a multiple of 32 dividing H, H a multiple of 32 (of 64
 * for 2-bit codes), variant in qsw_variant.  Pointers x, wg, wu, out must be
 * 16-byte aligned; scales/biases 2-byte aligned.  x and out must not overlap.
 * Rows M <= the small-M limit (qsw_set_gemv_max_m) run the memory-bound
 * kernel, the rest the tcgen05 tensor-core kernel; both compute the same
 * function.
 */
QSW_API qsw_status qswiglu_forward(const void *x, int64_t M, int64_t H, int64_t I,
                           const uint32_t *wg, const void *sg, const void *bg,
                           int gs_g, int bits_g,
                           const uint32_t *wu, const void *su, const void *bu,
                           int gs_u, int bits_u,
                           int variant, void *out, void *stream);

/*
 * Quantised linear y[M,N] = bf16(x[M,K] . W^T), W packed [N, K*bits/32]
 * with scales/biases [N, K/gs] (steel-linear-kernel.ts, steelLinear(): float
 * accumulator cast to bf16 at the store).  Used for the unfused comparison
 * path and for down_proj.  Same accepted shapes and alignment as above with
 * (H, I) -> (K, N).
 */
QSW_API qsw_status affine_qmm(const void *x, int64_t M, int64_t K, int64_t N,
                      const uint32_t *w, const void *s, const void *b,
                      int gs, int bits, void *y, void *stream);

/* Stream-K scheduling of the tensor-core kernel (qsw_set_stream_k). */
typedef enum {
    QSW_STREAM_K_OFF = 0,     /* whole output tiles, round-robin over the SMs */
    QSW_STREAM_K_AUTO = 1,    /* split K ranges where whole tiles would leave SMs idle (default) */
    QSW_STREAM_K_ALWAYS = 2   /* split whenever the tile count is not a multiple of the SM count */
} qsw_stream_k_mode;

/*
 * Bytes of workspace the *_ws entry points need on the current device
 * (a 1 KB header plus a 128 KB f32 partial accumulator per SM; 0 when no
 * device is current).
 */
QSW_API size_t qsw_workspace_bytes(void);

/*
 * qswiglu_forward / affine_qmm with a caller-owned device workspace that lets
 * the tensor-core kernel split the K range of output tiles between SMs
 * (stream-K) when whole tiles would fill the SMs unevenly -- e.g. 256 tiles on
 * 152 SMs.  A split tile is finished by the CTA holding its first K steps,
 * which adds the f32 partial accumulators that the others publish in the
 * workspace before the epilogue; results are the same function as the plain
 * entry points (f32 sums in a different order).
 *   workspace        device pointer, 256-byte aligned, zero-filled before its
 *                    first use (e.g. cudaMemsetAsync); the library keeps a
 *                    launch counter in it, so reuse it as is afterwards.  It
 *                    may be shared by the calls of one stream, not by calls
 *                    that can run concurrently.  NULL: whole tiles only.
 *   workspace_bytes  its size; less than qsw_workspace_bytes() returns
 *                    QSW_ERR_INVALID_ARG.
 * The small-M kernel does not use the workspace.  Other arguments, return
 * values and error behaviour as for the plain entry points.
 */
QSW_API qsw_status qswiglu_forward_ws(const void *x, int64_t M, int64_t H, int64_t I,
                           const uint32_t *wg, const void *sg, const void *bg,
                           int gs_g, int bits_g,
                           const uint32_t *wu, const void *su, const void *bu,
                           int gs_u, int bits_u,
                           int variant, void *out, void *workspace, size_t workspace_bytes,
                           void *stream);
QSW_API qsw_status affine_qmm_ws(const void *x, int64_t M, int64_t K, int64_t N,
                      const uint32_t *w, const void *s, const void *b,
                      int gs, int bits, void *y, void *workspace, size_t workspace_bytes,
                      void *stream);

/*
 * qswiglu_forward with stream-K scheduling and no caller workspace: the
 * split-tile partials go to a static device array of the library (sized for up
 * to 192 SMs; more SMs run whole tiles only), so the call allocates nothing
 * and takes no workspace argument.  The array is one per device: calls through
 * this entry point must not run concurrently with each other (use one stream,
 * or the *_ws form with one workspace per stream).  The first call on a device
 * also resolves the array's address and enqueues a 4 KB memset of its header
 * on `stream`; made inside a CUDA-graph capture, that memset becomes part of
 * the graph (every replay re-zeroes the header, which is harmless: the header
 * only needs to start at zero).  Should that first set-up fail, the call
 * returns QSW_ERR_CUDA and the next call tries again.  Arguments, results and
 * errors as for qswiglu_forward.
 */
QSW_API qsw_status qswiglu_forward_noalloc(const void *x, int64_t M, int64_t H, int64_t I,
                           const uint32_t *wg, const void *sg, const void *bg,
                           int gs_g, int bits_g,
                           const uint32_t *wu, const void *su, const void *bu,
                           int gs_u, int bits_u,
                           int variant, void *out, void *stream);

/*
 * The general forms: qswiglu_forward_ws / affine_qmm_ws / qsw_silu_mul with an
 * activation dtype (qsw_act_dtype; anything else returns QSW_ERR_INVALID_ARG).
 * With QSW_ACT_F16, x, scales, biases and the result are IEEE binary16 bit
 * patterns (same layouts and alignment), the dequantised weights are
 * f16(s*q + b) and the tensor cores run on f16 operands; everything else
 * (arguments, workspace, results, errors) is as for the bf16 forms.
 * affine_qmm_ex also takes `residual`: NULL, or [M, N] in the activation dtype
 * (16-byte aligned) added to the f32 accumulator before the one rounding,
 * y = T(x . W^T + residual); it may be y itself (each element is read before
 * it is written, by the same thread).
 */
QSW_API qsw_status qswiglu_forward_ex(const void *x, int64_t M, int64_t H, int64_t I,
                           const uint32_t *wg, const void *sg, const void *bg,
                           int gs_g, int bits_g,
                           const uint32_t *wu, const void *su, const void *bu,
                           int gs_u, int bits_u,
                           int variant, int act_dtype, void *out,
                           void *workspace, size_t workspace_bytes, void *stream);
QSW_API qsw_status affine_qmm_ex(const void *x, int64_t M, int64_t K, int64_t N,
                      const uint32_t *w, const void *s, const void *b,
                      int gs, int bits, int act_dtype, const void *residual, void *y,
                      void *workspace, size_t workspace_bytes, void *stream);
QSW_API qsw_status qsw_silu_mul_ex(const void *g, const void *u, int64_t n, int variant,
                        int act_dtype, void *out, void *stream);

/*
 * The whole MLP block with its residual (fused-mlp-kernel.ts on the pages:
 * the output is h + mlp(x)):
 *     hidden[M, I] = the fused expansion of x (variant QSW_MATCH or QSW_F32),
 *     y[M, Ho]     = T( h + hidden . Wd^T ),
 * down weights Wd packed [Ho, I*bits_d/32] with scales/biases [Ho, I/gs_d].
 * Two launches on `stream`: the fused expansion writes `hidden` (caller-owned,
 * [M, I] in the activation dtype, 16-byte aligned), then the down projection
 * adds the residual `h` ([M, Ho], or NULL for none; it may be y) to its f32
 * accumulator before the one rounding: deterministic, no atomics.  I must meet
 * the K rules of affine_qmm for the down weights (multiple of 32 and of gs_d).
 * The workspace (optional, as for the *_ws forms) serves both launches.
 * Argument errors in either stage return before anything is launched.
 */
QSW_API qsw_status qsw_mlp_forward_ex(const void *x, const void *h, int64_t M, int64_t H,
                           int64_t I, int64_t Ho,
                           const uint32_t *wg, const void *sg, const void *bg, int gs_g, int bits_g,
                           const uint32_t *wu, const void *su, const void *bu, int gs_u, int bits_u,
                           const uint32_t *wd, const void *sd, const void *bd, int gs_d, int bits_d,
                           int variant, int act_dtype, void *hidden, void *y,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Stream-K mode of the *_ws, *_ex and _noalloc entry points (qsw_stream_k_mode, default
 * QSW_STREAM_K_AUTO; other values are ignored).  Process-wide. */
QSW_API void qsw_set_stream_k(int mode);
QSW_API int qsw_get_stream_k(void);

/*
 * Elementwise out[i] = silu(g[i]) * u[i] over n bf16 values, the last step of
 * the unfused path (qwen3.ts, Qwen3MLP.forward: sigmoid, mul, mul).
 * variant QSW_MATCH rounds sigma, silu and the product to bf16; QSW_F32 rounds
 * once.  n >= 0; g, u, out 16-byte aligned; out may alias g or u.
 */
QSW_API qsw_status qsw_silu_mul(const void *g, const void *u, int64_t n, int variant,
                        void *out, void *stream);

/* Synchronise `stream`, then read and clear the device error word.
 * Returns QSW_ERR_BOUNDS if a debug-build check failed (libqswiglu_debug.so
 * only), else QSW_ERR_TIMEOUT if any kernel gave up on a wait since the last
 * call, QSW_ERR_CUDA if synchronisation failed, else QSW_OK. */
QSW_API qsw_status qsw_check_device_errors(void *stream);

/* 1 in the debug build (libqswiglu_debug.so, compiled with QSW_DEBUG_BOUNDS):
 * every kernel fills its shared-memory staging areas -- and the tensor-core
 * kernel its TMEM accumulators -- with NaN bit patterns at start, so a read of
 * staging data that was never written shows up as NaN in the results, and
 * checks TMA copy coordinates (16-byte innermost offsets), shared-memory
 * ranges and output indices, reporting a failure as QSW_ERR_BOUNDS through
 * qsw_check_device_errors() without trapping.  0 in the regular build. */
QSW_API int qsw_debug_build(void);

/* Largest M routed to the small-M kernels (default 32; 0 sends every M to the
 * tensor-core kernel).  Values above 32 are clamped to 32.  Process-wide. */
QSW_API void qsw_set_gemv_max_m(int m);
QSW_API int qsw_get_gemv_max_m(void);

/* Which small-M kernel serves a call routed to the small-M path. */
typedef enum {
    QSW_SMALL_M_AUTO = 0,   /* the warp-streamed kernel where it applies (H <= 16384 and its staging
                               fits in shared memory; M > 16 runs as launches over row chunks of 16,
                               each streaming the weights once), else the slot-ring kernel (default) */
    QSW_SMALL_M_RING = 1,   /* always the slot-ring kernel (bulk copies into shared-memory slots
                               shared by a CTA's warps) */
    QSW_SMALL_M_STREAM = 2  /* the warp-streamed kernel where it applies (each warp copies its own
                               blocks into a private ring), else the slot-ring one */
} qsw_small_m_kernel;

/* Selects the small-M kernel (qsw_small_m_kernel; other values are ignored).
 * Both compute the same function; the choice changes only which one runs and,
 * within the f32 accumulation bound, the order of the additions.
 * Process-wide. */
QSW_API void qsw_set_small_m_kernel(int kernel);
QSW_API int qsw_get_small_m_kernel(void);

/* Early weight stream (default off).  When on, the small-M kernels are
 * launched as programmatic dependents of the work before them on the stream:
 * a call may start while the previous kernel is still running and requests
 * the packed weights (and, on the slot-ring kernel, the scales and biases) of
 * its first units or K blocks into shared memory at once; it reads x and
 * writes its output only after all earlier work on the stream has completed
 * (griddepcontrol.wait).  Turn it on only when no earlier work on the stream
 * writes the weight, scale or bias arrays of the call -- the usual decode loop,
 * where weights are constant.  Process-wide. */
QSW_API void qsw_set_early_weight_stream(int on);
QSW_API int qsw_get_early_weight_stream(void);

/* Per-wait limit for device-side waits, in nanoseconds (default 4e9). */
QSW_API void qsw_set_wait_timeout_ns(uint64_t ns);

/* Test hook, not for production use: the next call served by the slot-ring
 * small-M kernel (the warp-streamed kernel has no spin waits) never requests the first unit of each of its CTAs, so every wait on
 * that unit's shared-memory slot runs out after the qsw_set_wait_timeout_ns
 * limit.  The kernel then lets its other copies land and returns without
 * writing its output, and the next qsw_check_device_errors() returns
 * QSW_ERR_TIMEOUT.  Later calls are unaffected.  Nothing traps and nothing
 * waits without a limit. */
QSW_API void qsw_debug_withhold_next_fill(void);

/* Dispatch counters (process-wide, monotonically increasing). `out` receives
 * min(n, QSW_NUM_COUNTERS) values. */
QSW_API void qsw_get_counters(uint64_t *out, int n);
QSW_API void qsw_reset_counters(void);

/* Static string for a status code. */
QSW_API const char *qsw_status_string(qsw_status s);

/* Library ABI version (major*100 + minor). */
QSW_API int qsw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSWIGLU_H_ */
