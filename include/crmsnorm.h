/*
 * crmsnorm.h -- C ABI of the GB300 (sm_103a) RMSNorm library.
 *
 * Row-wise RMSNorm forward (plain, fused residual add, Gemma w+1, FP32
 * zero-centred weight), its FP8 epilogues (static scale, 1x128 blocks), the
 * AdaRMSNorm style epilogues, RMSNorm + SiLU, LayerNorm (BF16 and FP8
 * output), and the training backward (dx and a deterministic FP32 dw).
 *
 * Sources cited below:
 *   [API]   "flashinfer.norm" API index (docs.flashinfer.ai/api/norm.html)
 *   [GUIDE] "FlashInfer normalization operator guide" article (sheratonhq.com),
 *           sections 2.1-2.4, 3.1-3.3, 6.1-6.5
 *   [CAKE]  "cake_rmsnorm_det_train_forward" reference page: Parameters,
 *           Returns, Notes
 *   [ADA]   "flashrt-adaptive-norms" README: formula block, Tensor Conventions
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, never synchronises, and enqueues its kernels on
 *     `stream` (0 = the legacy default stream) of the current device.
 *   - BF16 tensors are [T, H] row-major with a contiguous feature dimension
 *     and a row stride ld* given in ELEMENTS (ld >= H when T > 1).  Row
 *     strides let a [T, heads, H] slice of a wider [T, heads, W] buffer be
 *     normalised in place as T*heads rows of stride W.
 *   - Alignment: the fast path needs every BF16 base pointer 16-byte aligned,
 *     every row stride and H multiples of 8, FP32 weights 16-byte aligned and
 *     FP8 outputs 8-byte aligned; otherwise a 4-byte path needs BF16 bases
 *     4-byte aligned, even strides and an even H (FP32 weights 8-byte, FP8
 *     outputs 2-byte aligned).  Anything else returns CRMSN_ERR_ALIGNMENT.
 *   - Arithmetic: BF16 inputs, FP32 statistics with IEEE square root and
 *     division (no fast math), one rounding to the output format.
 *   - Every argument is checked before anything is enqueued; on an error
 *     nothing is launched.  T == 0 returns CRMSN_OK without a launch (row
 *     pointers may then be NULL; rmsnorm_bwd still zeroes dw).
 *   - In-place use: an output may be the very same tensor (same pointer and
 *     stride) as the input it replaces, as listed per function.  Any other
 *     overlap between an output and another tensor returns CRMSN_ERR_ALIAS.
 *   - The functions are safe to call from several host threads; kernels on
 *     one stream run in order.
 *   - Kernels are launched with programmatic dependent launch allowed, so a
 *     grid may be scheduled while the kernel before it in the stream is
 *     still running; each one waits (griddepcontrol.wait) for that kernel to
 *     complete before it touches memory.  A caller's own kernel launched
 *     with that attribute right after one of these must wait the same way
 *     before reading their outputs.
 */
#ifndef CRMSNORM_H
#define CRMSNORM_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

/* The library is built with hidden symbols; only these declarations are
 * exported. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum crmsn_status {
    CRMSN_OK = 0,
    CRMSN_ERR_NULL = 1,           /* a required pointer is NULL */
    CRMSN_ERR_SHAPE = 2,          /* T < 0, H < 1, odd H where H must be even, ld < H */
    CRMSN_ERR_UNSUPPORTED_H = 3,  /* H outside the supported range of the operation */
    CRMSN_ERR_ALIGNMENT = 4,      /* pointer or stride alignment (see above) */
    CRMSN_ERR_DTYPE = 5,          /* unknown weight dtype or FP8 kind */
    CRMSN_ERR_WORKSPACE = 6,      /* backward workspace too small or misaligned */
    CRMSN_ERR_ALIAS = 7,          /* outputs overlap inputs other than as allowed */
    CRMSN_ERR_CUDA = 8,           /* the CUDA runtime reported an error */
    CRMSN_ERR_DEVICE_TIMEOUT = 9, /* reserved: the kernels have no device-side waits */
    CRMSN_ERR_ARG = 10,           /* eps / scale value out of range */
    CRMSN_ERR_SCRATCH_LIMIT = 11, /* rmsnorm_bwd_noalloc: problem needs more than its built-in scratch */
    CRMSN_ERR_NOT_DEBUG_BUILD = 12 /* crmsn_debug_status: the library has no bounds guard */
} crmsn_status;

/* Weight storage types. */
enum { CRMSN_BF16 = 0, CRMSN_F32 = 1 };
/* FP8 output formats. */
enum { CRMSN_E4M3 = 0, CRMSN_E5M2 = 1 };
/* Output formats of fused_rmsnorm_silu. */
enum { CRMSN_OUT_BF16 = 0, CRMSN_OUT_E4M3 = 1 };
/* Operation ids for rmsnorm_supports(). */
enum {
    CRMSN_OP_FWD = 0,
    CRMSN_OP_BWD = 1,
    CRMSN_OP_QUANT = 2,
    CRMSN_OP_BLOCK_QUANT = 3,
    CRMSN_OP_ADA_STYLE = 4,
    CRMSN_OP_GATED_ADA_FP8 = 5,
    CRMSN_OP_SILU = 6,
    CRMSN_OP_LAYERNORM = 7
};

/* Largest supported hidden size. */
#define CRMSN_MAX_H 16384

/*
 * rmsnorm_fwd -- [API] rmsnorm, gemma_rmsnorm, fused_add_rmsnorm,
 * gemma_fused_add_rmsnorm; [GUIDE] 2.1-2.2, 3.1, 6.1; [CAKE] Parameters and
 * Returns.
 *
 *   residual == NULL:  h = x
 *   residual != NULL:  h = h_new = bf16(x + residual)    (written to h_new)
 *   rstd[t] = 1 / sqrt(mean_j h[t,j]^2 + eps)            (FP32, nullable)
 *   y[t,j]  = bf16((h[t,j] * rstd[t]) * w_eff[j])
 *   w_eff   = f32(w + weight_bias); w is BF16 or FP32 (w_dtype).  Gemma is
 *             weight_bias = 1 on a BF16 weight; the zero-centred FP32 weight
 *             of [CAKE] is weight_bias = 1 on an FP32 weight.
 *
 * x, residual, y, h_new: BF16 [T, H] with row strides ldx, ldr, ldy, ldh.
 * w: [H] contiguous.  rstd: FP32 [T] or NULL.  h_new is required iff
 * residual is given.  In place: y == x (same ldy == ldx) and
 * h_new == residual (ldh == ldr) are allowed; that pair of calls is
 * fused_add_rmsnorm.  Supports 1 <= H <= CRMSN_MAX_H.
 */
crmsn_status rmsnorm_fwd(const void *x, int64_t ldx,
                         const void *residual, int64_t ldr,
                         const void *w, int w_dtype, float weight_bias,
                         float eps, int64_t T, int64_t H,
                         void *y, int64_t ldy, float *rstd,
                         void *h_new, int64_t ldh, cudaStream_t stream);

/*
 * rmsnorm_bwd -- [API] cake_rmsnorm_train_backward; [GUIDE] 6.1-6.3;
 * [CAKE] Notes (deterministic dw).
 *
 *   m[t]     = mean_j g[t,j] * w_eff[j] * x[t,j]
 *   dx[t,j]  = bf16(rstd[t]*g[t,j]*w_eff[j] - x[t,j]*rstd[t]^3*m[t]
 *                   (+ g_residual[t,j]))
 *   dw[j]    = sum_t g[t,j] * x[t,j] * rstd[t]            (FP32, overwritten)
 *
 * x is the tensor the forward normalised (h_new on the residual route) and
 * rstd the forward's FP32 output.  g_residual (nullable) is the gradient
 * arriving directly at h_new; dx is then the gradient of both residual-add
 * inputs.  g, x, g_residual, dx: BF16 [T, H] with row strides.  w as in
 * rmsnorm_fwd.  dw: FP32 [H].  In place: dx == g (lddx == ldg) is allowed.
 *
 * dw is reduced deterministically.  Up to 2048 rows (the column form, one
 * launch): fixed strips of columns are each summed over all rows in a fixed
 * order with compensated FP32 sums, the order depending only on T, H and the
 * access width (the 16-byte or the 4-byte path), not on the SM count; the
 * workspace is not touched.  Above 2048 rows: rows are cut into a fixed
 * table of contiguous chunks (a function of T and the device's SM count),
 * each chunk sums its rows in a fixed order with compensated FP32 sums into
 * the workspace, and a second kernel adds the chunk sums in a fixed order,
 * so the same T on devices with the same SM count gives the same dw bits.
 * dx does not depend on the form or the chunk table.
 * workspace: caller-owned device memory of at least
 * rmsnorm_bwd_workspace_bytes() bytes, 256-byte aligned, any initial
 * content; it is scratch only and may be reused by any later call on the
 * same stream.  T == 0 writes dw = 0 (a memset) and launches no kernel.
 */
crmsn_status rmsnorm_bwd(const void *g, int64_t ldg,
                         const void *x, int64_t ldx,
                         const void *w, int w_dtype, float weight_bias,
                         const float *rstd,
                         const void *g_residual, int64_t ldgr,
                         int64_t T, int64_t H,
                         void *dx, int64_t lddx, float *dw,
                         void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * rmsnorm_bwd_workspace_bytes -- [API]
 * cake_rmsnorm_train_backward_workspace_bytes; [GUIDE] 6.3.
 * Bytes of backward workspace for width H on `device`: FP32 partial dw rows,
 * one per chunk, sized for the device's largest chunk count, so the value
 * does not depend on `rows`; `residual` is accepted for signature parity and
 * does not change the size.  Returns 0 for an invalid H or device.
 */
size_t rmsnorm_bwd_workspace_bytes(int64_t rows, int64_t H, int device,
                                   int residual);

/*
 * rmsnorm_bwd_noalloc -- no counterpart on the pages: the backward of
 * rmsnorm_bwd for callers that cannot provide a workspace (engines and plugin
 * hosts that plan all device memory in advance and forbid allocation inside
 * an operation, or C callers without a device allocator, for whom a
 * cudaMalloc per call would also stall the device).  Same arguments, results
 * and dw determinism as rmsnorm_bwd, minus the workspace; allocates nothing.
 *
 * The scratch is a 16 MiB array in the library's own device memory, held by
 * every GPU that loads the library until the process exits.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress with
 * that device current); make that first call before any stream capture.  The
 * address is kept per device number for the life of the process, so it is
 * only valid in the context that made the first call: calls after
 * cudaDeviceReset on that device, or from a context other than the device's
 * primary context (the one the runtime API uses), are not supported.  All
 * calls on a device share the array: calls that overlap on the GPU (other
 * streams or host threads) race and must be serialised.  The scratch needs
 * no zeroing.  Problems whose workspace (rmsnorm_bwd_workspace_bytes) exceeds
 * 16 MiB return CRMSN_ERR_SCRATCH_LIMIT without launching anything; on a
 * 152-SM GB300 every H fits (the workspace stays below 12 MB).
 */
crmsn_status rmsnorm_bwd_noalloc(const void *g, int64_t ldg,
                                 const void *x, int64_t ldx,
                                 const void *w, int w_dtype, float weight_bias,
                                 const float *rstd,
                                 const void *g_residual, int64_t ldgr,
                                 int64_t T, int64_t H,
                                 void *dx, int64_t lddx, float *dw,
                                 cudaStream_t stream);

/*
 * fused_add_rmsnorm_quant -- [API] fused_add_rmsnorm_quant and rmsnorm_quant;
 * [GUIDE] 3.2.
 *
 *   residual != NULL:  residual <- h = bf16(x + residual)   (in place)
 *   residual == NULL:  h = x                                (rmsnorm_quant)
 *   out[t,j] = fp8(f32((h*rstd)*w_eff) / scale[0])   round to nearest even,
 *              saturating to the largest finite FP8 value
 *
 * out: FP8 [T, H] (E4M3FN or E5M2 by fp8_kind) with row stride ldo (bytes =
 * elements).  scale: device pointer to one FP32 value (> 0).  rstd: FP32
 * [T] or NULL.  x, residual: BF16 with row strides ldx, ldr.
 */
crmsn_status fused_add_rmsnorm_quant(void *out, int64_t ldo, int fp8_kind,
                                     const void *x, int64_t ldx,
                                     void *residual, int64_t ldr,
                                     const void *w, int w_dtype,
                                     float weight_bias, const float *scale,
                                     float eps, int64_t T, int64_t H,
                                     float *rstd, cudaStream_t stream);

/*
 * fused_add_rmsnorm_fp8_block_quant -- [API] same name; [GUIDE] 3.3.
 *
 *   residual <- h = bf16(x + residual)                       (in place)
 *   normed_out[t,j] = n = bf16((h*rstd)*w[j])
 *   per row t and 128-column block b:
 *     s = f32(max_{j in b} |n[t,j]| / 448)
 *     out[t,j] = e4m3(f32(n[t,j] / s))        (0 when s == 0)
 *     block_scale[b * ldT + t] = s
 *
 * out: E4M3FN [T, H] contiguous; normed_out: BF16 [T, H] contiguous;
 * block_scale: FP32 (H/128) x ldT column-major ("MN-major"), ldT >= T
 * (the pages use round_up(T, 4)); columns t >= T are not written.
 * x, residual: BF16 with row strides ldx, ldr.  w: BF16 [H].
 * H must be a multiple of 128 and at most CRMSN_MAX_H, else
 * CRMSN_ERR_UNSUPPORTED_H.
 */
crmsn_status fused_add_rmsnorm_fp8_block_quant(void *out, float *block_scale,
                                               int64_t ldT, void *normed_out,
                                               const void *x, int64_t ldx,
                                               void *residual, int64_t ldr,
                                               const void *w, float eps,
                                               int64_t T, int64_t H,
                                               cudaStream_t stream);

/*
 * ada_rms_norm_style -- [ADA] ada_rms_norm_style_bf16, formula block and
 * Tensor Conventions.
 *
 *   o = (x*rstd)*w;  out = bf16(o * (1 + style[s, 0:D]) + style[s, D:2D])
 *   gate_out = style[s, 2D:3D]                (bit copy)
 *   s = t when style_rows == T, s = 0 when style_rows == 1 (broadcast; the
 *   row is read directly, never materialised).
 *
 * x, out, gate_out: BF16 [T, D] contiguous; style: BF16 [style_rows, 3D]
 * contiguous; w: BF16 [D].  D must be even (CRMSN_ERR_SHAPE otherwise).
 */
crmsn_status ada_rms_norm_style(const void *x, const void *w,
                                const void *style, int64_t style_rows,
                                float eps, int64_t T, int64_t D,
                                void *out, void *gate_out, cudaStream_t stream);

/*
 * gate_residual_ada_norm_fp8 -- [ADA] gate_residual_ada_norm_fp8_static_bf16.
 *
 *   residual <- h = bf16(residual + bf16(x * gate))       (in place)
 *   o = (h*rstd)*w;  v = f32(o * (1 + sc) + sh)
 *   out = e4m3(f32(v / scale[0]))             (round to nearest even, saturating)
 *   gate_out = style[s, 2D:3D]
 *
 * residual, x, gate, gate_out: BF16 [T, D] contiguous; out: E4M3FN [T, D]
 * contiguous; style as in ada_rms_norm_style; scale: device FP32 [1].
 */
crmsn_status gate_residual_ada_norm_fp8(void *residual, const void *x,
                                        const void *gate, const void *w,
                                        const void *style, int64_t style_rows,
                                        const float *scale, float eps,
                                        int64_t T, int64_t D,
                                        void *out, void *gate_out,
                                        cudaStream_t stream);

/*
 * fused_rmsnorm_silu -- [API] fused_rmsnorm_silu; [GUIDE] 5.1.
 *
 *   v[t,j] = (x[t,j] * rstd[t]) * w_eff[j]   (the plain rmsnorm_fwd value)
 *   s      = SiLU(v) = v / (1 + exp(-v))    (FP32; see the error note below)
 *   CRMSN_OUT_BF16: out = bf16(s)
 *   CRMSN_OUT_E4M3: out = e4m3(s / scale), saturating to +-448; scale is a
 *                   device FP32 [1] or NULL for no scale (the guide names none)
 *
 * x: BF16 [T, H], row stride ldx.  out: BF16 or E4M3FN [T, H], row stride
 * ldo; a BF16 out may be x itself (same pointer and stride).  w: BF16 or FP32
 * [H] (w_dtype) with weight_bias as in rmsnorm_fwd.  rstd: FP32 [T] or NULL.
 * SiLU uses the fast exponential and reciprocal: its relative error is about
 * 2^-20 where |v| < 10 and stays far below a BF16 half-ulp everywhere.  The
 * guide's NVFP4 output is not provided.  Errors: CRMSN_ERR_DTYPE for another
 * out_format or w_dtype; the rest as rmsnorm_fwd.  1 <= H <= CRMSN_MAX_H, H
 * even.
 */
crmsn_status fused_rmsnorm_silu(void *out, int64_t ldo, int out_format,
                                const void *x, int64_t ldx,
                                const void *w, int w_dtype, float weight_bias,
                                const float *scale, float eps,
                                int64_t T, int64_t H, float *rstd,
                                cudaStream_t stream);

/*
 * layernorm -- [API] layernorm; [GUIDE] 4.
 *
 *   mean[t] = (1/H) sum_j x[t,j]
 *   var[t]  = (1/H) sum_j (x[t,j] - mean[t])^2       (population variance)
 *   rstd[t] = 1 / sqrt(var[t] + eps)
 *   y[t,j]  = bf16((x[t,j] - mean[t]) * rstd[t] * gamma[j] + beta[j])
 *
 * x, y: BF16 [T, H] with row strides ldx, ldy; y may be x itself (same
 * pointer and stride).  gamma, beta: FP32 [H], contiguous (the guide's
 * "gemma" is gamma).  mean, rstd: FP32 [T] or NULL (FP32 statistics, the
 * mean summed and the deviations squared in FP32 with compensated sums across
 * threads).  Errors as rmsnorm_fwd; 1 <= H <= CRMSN_MAX_H, H even.
 */
crmsn_status layernorm(void *y, int64_t ldy, const void *x, int64_t ldx,
                       const float *gamma, const float *beta, float eps,
                       int64_t T, int64_t H, float *mean, float *rstd,
                       cudaStream_t stream);

/*
 * layernorm_quant -- [API] layernorm_quant; [GUIDE] 4.
 *
 *   out[t,j] = fp8(((x - mean) * rstd * gamma + beta) / scale)
 *
 * as layernorm, with the value divided by the device FP32 scale [1] before
 * the cast to E4M3FN or E5M2 (fp8_kind), saturating.  out: [T, H] bytes with
 * row stride ldo.  Errors: CRMSN_ERR_DTYPE for another fp8_kind,
 * CRMSN_ERR_NULL for a NULL scale; the rest as layernorm.
 */
crmsn_status layernorm_quant(void *out, int64_t ldo, int fp8_kind,
                             const void *x, int64_t ldx,
                             const float *gamma, const float *beta,
                             const float *scale, float eps,
                             int64_t T, int64_t H, float *mean, float *rstd,
                             cudaStream_t stream);

/*
 * crmsn_debug_status -- no counterpart on the pages: the bounds guard of the
 * debug build (compiled with -DCRMSN_DEBUG; build.py's debug option).  In
 * that build every global load and store of every kernel is checked against
 * the byte ranges of the call's tensors (all readable; outputs and the
 * workspace writable) and every dynamic shared-memory access against the
 * launch's size; an access outside them is skipped (a load reads zeros) and
 * the first one is recorded.  This call waits for the device
 * (cudaDeviceSynchronize), stores the recorded word in *violation (0 when
 * every access was in bounds; otherwise bit 63 set, bits 62..56 the kind --
 * 1 load, 2 store, 3 asynchronous copy, 4 shared memory -- bits 55..32 the
 * CTA, 31..22 the thread, 21..0 the low bits of the global address or of
 * the shared-memory byte offset) and clears it.  The
 * normal build stores 0 and returns CRMSN_ERR_NOT_DEBUG_BUILD.
 */
crmsn_status crmsn_debug_status(uint64_t *violation);

/*
 * rmsnorm_supports -- [API] supports_* helpers; [GUIDE] 6.1
 * is_cake_rmsnorm_train_supported.  CRMSN_OK when operation `op` (CRMSN_OP_*)
 * accepts hidden size H with weight dtype w_dtype, else the status the call
 * would return for that H / dtype.
 */
crmsn_status rmsnorm_supports(int64_t H, int w_dtype, int op);

/* Human-readable name of a status. */
const char *crmsn_status_str(crmsn_status status);

#ifdef __cplusplus
}
#endif

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#endif /* CRMSNORM_H */
