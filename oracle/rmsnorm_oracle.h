/*
 * rmsnorm_oracle.h -- plain, single-threaded FP64 CPU oracle for row-wise RMSNorm.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline call this library. It shares no code, header, table or helper with
 * the CUDA library and never includes anything from it.
 *
 * Storage conventions
 *   BF16 values travel as their raw 16-bit patterns (uint16_t), FP8 E4M3FN /
 *   E5M2 values as raw 8-bit codes (uint8_t), FP32 values as float.
 *   Row strides (ld*) are in elements.  Outputs are written row-major and
 *   contiguous ([T, H], leading dimension H) unless stated.  Every "exact"
 *   output is the double-precision value before the final rounding; rounded
 *   outputs use this file's own codecs.
 *
 * Sources (cited per function in the .c file)
 *   [API]   "flashinfer.norm" API index, docs.flashinfer.ai/api/norm.html
 *   [GUIDE] "FlashInfer normalization operator guide" article (sheratonhq.com),
 *           sections 2.1-2.4, 3.1-3.3, 4, 6.1-6.5
 *   [CAKE]  "cake_rmsnorm_det_train_forward" reference page: Parameters,
 *           Returns, Notes
 *   [ADA]   "flashrt-adaptive-norms" README: overview formula block, Tensor
 *           Conventions, Validation
 */
#ifndef RMSNORM_ORACLE_H
#define RMSNORM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
double   orc_bf16_to_f64(uint16_t bits);
uint16_t orc_bf16_from_f64(double v);          /* round to nearest, ties to even */
double   orc_e4m3_to_f64(uint8_t code);
uint8_t  orc_e4m3_from_f32(float v);           /* RNE, saturate to +-448, NaN -> 0x7F */
double   orc_e5m2_to_f64(uint8_t code);
uint8_t  orc_e5m2_from_f32(float v);           /* RNE, saturate to +-57344, NaN -> 0x7F */
/* The same conversions applied elementwise to n values (fp8_kind 0 = E4M3FN,
 * 1 = E5M2). */
void orc_bf16_to_f64_n(int64_t n, const uint16_t *in, double *out);
void orc_bf16_from_f64_n(int64_t n, const double *in, uint16_t *out);
void orc_fp8_to_f64_n(int64_t n, int fp8_kind, const uint8_t *in, double *out);
void orc_fp8_from_f32_n(int64_t n, int fp8_kind, const float *in, uint8_t *out);

/* ---- the row math in double (no storage format involved) --------------- */
/* rstd = 1/sqrt(mean(h^2) + eps); yv[j] = h[j] * rstd * w_eff[j]. Returns rstd. */
double orc_row_fwd_f64(int64_t H, const double *h, const double *w_eff,
                       double eps, double *yv);
/* m = mean(g * w_eff * h);
 * dxv[j] = rstd*g[j]*w_eff[j] - h[j]*rstd^3*m (+ g_res[j] when g_res != NULL);
 * dw_row[j] = g[j]*h[j]*rstd (nullable).  Returns m. */
double orc_row_bwd_f64(int64_t H, const double *g, const double *h,
                       const double *w_eff, double rstd, const double *g_res,
                       double *dxv, double *dw_row);

/* ---- operations on stored tensors --------------------------------------- */
/* Effective weight w_eff[j] = f32(w[j] + weight_bias); w is BF16 bits
 * (w_is_f32 == 0) or float (w_is_f32 != 0). */
void orc_weight_eff(int64_t H, const void *w, int w_is_f32, float weight_bias,
                    double *w_eff);

/* RMSNorm forward, plain or with the fused residual add.
 * residual == NULL: h = x.  Otherwise h_new = bf16(x + residual) is written to
 * h_new (required) and normalised.  y_exact/y/rstd_exact/rstd32 are nullable. */
void orc_rmsnorm_fwd(int64_t T, int64_t H,
                     const uint16_t *x, int64_t ldx,
                     const uint16_t *residual, int64_t ldr,
                     const void *w, int w_is_f32, float weight_bias, float eps,
                     double *y_exact, uint16_t *y, double *rstd_exact,
                     float *rstd32, uint16_t *h_new);

/* RMSNorm backward for rows normalised with the saved FP32 rstd.
 * x is the tensor the forward normalised (h_new on the residual route).
 * g_res (nullable) is the gradient flowing straight into h_new.
 * Writes dx_exact (nullable), dx (nullable), m_out[T] (nullable),
 * dw[H] = sum_t g*x*rstd and dw_abs[H] = sum_t |g*x*rstd| (both nullable). */
void orc_rmsnorm_bwd(int64_t T, int64_t H,
                     const uint16_t *g, int64_t ldg,
                     const uint16_t *x, int64_t ldx,
                     const void *w, int w_is_f32, float weight_bias,
                     const float *rstd,
                     const uint16_t *g_res, int64_t ldgr,
                     double *dx_exact, uint16_t *dx, double *m_out,
                     double *dw, double *dw_abs);

/* (Fused add) RMSNorm + FP8 with a static scale: q = fp8(f32(yv / scale)).
 * residual == NULL is the plain rmsnorm_quant.  fp8_kind 0 = E4M3FN, 1 = E5M2.
 * v_exact (nullable) receives yv / scale before the FP32 decision.           */
void orc_rmsnorm_quant(int64_t T, int64_t H,
                       const uint16_t *x, int64_t ldx,
                       const uint16_t *residual, int64_t ldr,
                       const void *w, int w_is_f32, float weight_bias,
                       float scale, float eps, int fp8_kind,
                       uint16_t *h_new, double *v_exact, uint8_t *q,
                       float *rstd32);

/* Fused add + RMSNorm + 1x128 FP8 block quantisation.
 * normed = bf16(yv); per row and 128-column block b: s = f32(amax|normed|/448),
 * q = e4m3(f32(normed / s)) (all codes 0 when s == 0);
 * block_scale[b * ldT + t] = s for t < T (ldT >= T).                          */
void orc_fused_add_rmsnorm_fp8_block_quant(int64_t T, int64_t H,
                       const uint16_t *x, int64_t ldx,
                       const uint16_t *residual, int64_t ldr,
                       const uint16_t *w, float eps,
                       uint16_t *h_new, double *normed_exact, uint16_t *normed,
                       float *block_scale, int64_t ldT, uint8_t *q);

/* AdaRMSNorm with style (contiguous rows; style_rows is T or 1):
 * ov = yv * (1 + style[:, 0:D]) + style[:, D:2D]; out = bf16(ov);
 * gate_out = style[:, 2D:3D] (copied bits).                                   */
void orc_ada_rms_norm_style(int64_t T, int64_t D,
                            const uint16_t *x, const uint16_t *w,
                            const uint16_t *style, int64_t style_rows, float eps,
                            double *out_exact, uint16_t *out, uint16_t *gate_out);

/* Gated residual + AdaRMSNorm + static FP8:
 * residual_out = bf16(residual + bf16(x * gate)); normalise residual_out;
 * v = (yv * (1 + sc) + sh) / scale; q = e4m3(f32(v)); gate_out as above.       */
void orc_gate_residual_ada_norm_fp8(int64_t T, int64_t D,
                            const uint16_t *residual, const uint16_t *x,
                            const uint16_t *gate, const uint16_t *w,
                            const uint16_t *style, int64_t style_rows,
                            float scale, float eps,
                            uint16_t *residual_out, double *v_exact, uint8_t *q,
                            uint16_t *gate_out);

/* RMSNorm + SiLU: s = yv / (1 + exp(-yv)) of the plain forward's yv.
 * out_fp8 == 0: y = bf16(s), v_exact = s.  out_fp8 != 0: q = e4m3(f32(s /
 * scale)), v_exact = s / scale.  y or q may be NULL for the other output. */
void orc_fused_rmsnorm_silu(int64_t T, int64_t H,
                            const uint16_t *x, int64_t ldx,
                            const void *w, int w_is_f32, float weight_bias,
                            float eps, int out_fp8, float scale,
                            double *v_exact, uint16_t *y, uint8_t *q,
                            float *rstd32);

/* LayerNorm: o = (x - mean) * rstd * gamma + beta, rstd = 1/sqrt(var + eps),
 * var the population variance.  out_fp8 == 0: y = bf16(o), v_exact = o.
 * out_fp8 != 0: q = fp8(f32(o / scale)) (fp8_kind 0 E4M3FN, 1 E5M2),
 * v_exact = o / scale.  mean_out, rstd_out, v_exact nullable. */
void orc_layernorm(int64_t T, int64_t H,
                   const uint16_t *x, int64_t ldx,
                   const float *gamma, const float *beta, float eps,
                   int out_fp8, int fp8_kind, float scale,
                   double *v_exact, uint16_t *y, uint8_t *q,
                   double *mean_out, double *rstd_out);

#ifdef __cplusplus
}
#endif
#endif /* RMSNORM_ORACLE_H */
