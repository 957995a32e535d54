/*
 * rmsnorm_oracle.c -- plain, single-threaded FP64 CPU oracle for row-wise RMSNorm.
 *
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
 * baseline may call it.  It is written from the pages' definitions, evaluates
 * every statistic in double precision, and rounds only where the pages store a
 * value (BF16 outputs, the FP32 rstd, FP8 codes), with codecs written here from
 * the format definitions.  No blocking, fusion or reordering: each operation is
 * the loop over rows of the definition.  Build without -ffast-math and with
 * -ffp-contract=off so that x86_64 and aarch64 builds give the same bits.
 *
 * Source abbreviations are listed in rmsnorm_oracle.h.
 */
#include "rmsnorm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ========================================================================
 * Number formats
 * ======================================================================== */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits; the
 * upper half of an IEEE binary32.  Exponent field 0 holds zero and the
 * subnormals (fraction * 2^-133), 255 holds inf/NaN. */
double orc_bf16_to_f64(uint16_t bits)
{
    int s = bits >> 15;
    int e = (bits >> 7) & 0xFF;
    int f = bits & 0x7F;
    double v;
    if (e == 0xFF)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -126 - 7);
    else
        v = ldexp((double)(128 + f), e - 127 - 7);
    return s ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to the even significand.
 * The quantum at |v| in [2^E, 2^(E+1)) is 2^(E-7), and below the smallest
 * normal 2^-126 it stays 2^-133.  Results beyond the largest finite value
 * become infinity (IEEE round-to-nearest overflow). */
uint16_t orc_bf16_from_f64(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);             /* a = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;                  /* floor(log2 a) */
    if (E < -126)
        E = -126;
    double k = rint(ldexp(a, 7 - E)); /* significand in quanta; rint ties to even */
    if (k >= 256.0) {                /* rounded up into the next binade */
        k = 128.0;
        E += 1;
    }
    if (k < 128.0)                   /* subnormal: exponent field 0 */
        return sign | (uint16_t)k;
    if (E + 127 >= 255)
        return sign | 0x7F80;
    return sign | (uint16_t)(((E + 127) << 7) | ((int)k - 128));
}

/* OCP FP8 E4M3FN: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities, S.1111.111 is NaN, the largest finite value is 448 (0x7E);
 * subnormals are fraction * 2^-9. */
double orc_e4m3_to_f64(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int f = code & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 7 - 3);
    return s ? -v : v;
}

/* Round a float to E4M3FN, nearest with ties to even, saturating values whose
 * magnitude exceeds 448 (infinities included) to +-448; NaN becomes 0x7F. */
uint8_t orc_e4m3_from_f32(float vf)
{
    double v = (double)vf;
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= 448.0)
        return sign | 0x7E;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    if (E < -6)
        E = -6;
    double k = rint(ldexp(a, 3 - E));
    if (k >= 16.0) {
        k = 8.0;
        E += 1;
    }
    int code = (k < 8.0) ? (int)k : (((E + 7) << 3) | ((int)k - 8));
    if (code > 0x7E)
        code = 0x7E;
    return (uint8_t)(sign | code);
}

/* OCP FP8 E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits; exponent
 * field 31 holds inf (fraction 0) and NaN; the largest finite value is 57344
 * (0x7B); subnormals are fraction * 2^-16. */
double orc_e5m2_to_f64(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 2) & 0x1F;
    int f = code & 0x3;
    double v;
    if (e == 31)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -16);
    else
        v = ldexp((double)(4 + f), e - 15 - 2);
    return s ? -v : v;
}

/* Round a float to E5M2, nearest with ties to even, saturating magnitudes
 * above 57344 (infinities included) to +-57344; NaN becomes 0x7F. */
uint8_t orc_e5m2_from_f32(float vf)
{
    double v = (double)vf;
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= 57344.0)
        return sign | 0x7B;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    if (E < -14)
        E = -14;
    double k = rint(ldexp(a, 2 - E));
    if (k >= 8.0) {
        k = 4.0;
        E += 1;
    }
    int code = (k < 4.0) ? (int)k : (((E + 15) << 2) | ((int)k - 4));
    if (code > 0x7B)
        code = 0x7B;
    return (uint8_t)(sign | code);
}

/* Elementwise forms of the conversions above (fp8_kind 0 = E4M3FN, 1 = E5M2). */
void orc_bf16_to_f64_n(int64_t n, const uint16_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_to_f64(in[i]);
}

void orc_bf16_from_f64_n(int64_t n, const double *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_from_f64(in[i]);
}

void orc_fp8_to_f64_n(int64_t n, int fp8_kind, const uint8_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fp8_kind ? orc_e5m2_to_f64(in[i]) : orc_e4m3_to_f64(in[i]);
}

void orc_fp8_from_f32_n(int64_t n, int fp8_kind, const float *in, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fp8_kind ? orc_e5m2_from_f32(in[i]) : orc_e4m3_from_f32(in[i]);
}

/* ========================================================================
 * Row math in double
 * ======================================================================== */

/* [GUIDE] 2.1: out = input / RMS(input) * weight; [CAKE] Returns and [GUIDE]
 * 6.1: rstd = 1/sqrt(mean(h^2) + eps), eps added to the mean inside the root;
 * [GUIDE] 2.2 / 2.4: the weight enters as (w + weight_bias). */
double orc_row_fwd_f64(int64_t H, const double *h, const double *w_eff,
                       double eps, double *yv)
{
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j)
        ss += h[j] * h[j];
    double rstd = 1.0 / sqrt(ss / (double)H + eps);
    if (yv)
        for (int64_t j = 0; j < H; ++j)
            yv[j] = h[j] * rstd * w_eff[j];
    return rstd;
}

/* [GUIDE] 6.1: dx = r*g*w - x*r^3*mean(g*w*x) and dw = sum_t g*x*r;
 * [GUIDE] 6.2: with g_residual the returned dx also carries the gradient that
 * flows straight into h_new, so it is added to the normalisation gradient. */
double orc_row_bwd_f64(int64_t H, const double *g, const double *h,
                       const double *w_eff, double rstd, const double *g_res,
                       double *dxv, double *dw_row)
{
    double dot = 0.0;
    for (int64_t j = 0; j < H; ++j)
        dot += g[j] * w_eff[j] * h[j];
    double m = dot / (double)H;
    double r3 = rstd * rstd * rstd;
    for (int64_t j = 0; j < H; ++j) {
        double d = rstd * g[j] * w_eff[j] - h[j] * r3 * m;
        if (g_res)
            d += g_res[j];
        if (dxv)
            dxv[j] = d;
        if (dw_row)
            dw_row[j] = g[j] * h[j] * rstd;
    }
    return m;
}

/* [GUIDE] 2.2: Gemma uses w + 1 through weight_bias; [CAKE] Parameters/w: an
 * FP32 weight is the zero-centred form whose effective weight 1 + w the model
 * computes in FP32.  Both are the FP32 sum f32(w + bias); the double sum of two
 * floats rounded once to float is that correctly rounded FP32 sum. */
void orc_weight_eff(int64_t H, const void *w, int w_is_f32, float weight_bias,
                    double *w_eff)
{
    for (int64_t j = 0; j < H; ++j) {
        double wj = w_is_f32 ? (double)((const float *)w)[j]
                             : orc_bf16_to_f64(((const uint16_t *)w)[j]);
        w_eff[j] = (double)(float)(wj + (double)weight_bias);
    }
}

/* Load row t of the normalised input into h (double).  residual == NULL: the
 * input itself.  Otherwise [GUIDE] 3.1 / [CAKE] Parameters/x: the residual
 * stream update h_new = bf16(x + residual), stored and then normalised. */
static void load_row(int64_t t, int64_t H, const uint16_t *x, int64_t ldx,
                     const uint16_t *residual, int64_t ldr, double *h,
                     uint16_t *h_new)
{
    for (int64_t j = 0; j < H; ++j) {
        double xj = orc_bf16_to_f64(x[t * ldx + j]);
        if (residual) {
            double uj = orc_bf16_to_f64(residual[t * ldr + j]);
            uint16_t hn = orc_bf16_from_f64(xj + uj);
            if (h_new)
                h_new[t * H + j] = hn;
            h[j] = orc_bf16_to_f64(hn);
        } else {
            h[j] = xj;
        }
    }
}

/* ========================================================================
 * Operations
 * ======================================================================== */

/* [API] rmsnorm / gemma_rmsnorm / fused_add_rmsnorm; [CAKE] forward:
 * y = bf16((h * rstd) * w_eff), one FP32 rstd per row. */
void orc_rmsnorm_fwd(int64_t T, int64_t H,
                     const uint16_t *x, int64_t ldx,
                     const uint16_t *residual, int64_t ldr,
                     const void *w, int w_is_f32, float weight_bias, float eps,
                     double *y_exact, uint16_t *y, double *rstd_exact,
                     float *rstd32, uint16_t *h_new)
{
    double *h = malloc(sizeof(double) * (size_t)H);
    double *we = malloc(sizeof(double) * (size_t)H);
    double *yv = malloc(sizeof(double) * (size_t)H);
    orc_weight_eff(H, w, w_is_f32, weight_bias, we);
    for (int64_t t = 0; t < T; ++t) {
        load_row(t, H, x, ldx, residual, ldr, h, h_new);
        double r = orc_row_fwd_f64(H, h, we, (double)eps, yv);
        for (int64_t j = 0; j < H; ++j) {
            if (y_exact)
                y_exact[t * H + j] = yv[j];
            if (y)
                y[t * H + j] = orc_bf16_from_f64(yv[j]);
        }
        if (rstd_exact)
            rstd_exact[t] = r;
        if (rstd32)
            rstd32[t] = (float)r;
    }
    free(h);
    free(we);
    free(yv);
}

/* [GUIDE] 6.1-6.2 backward with the FP32 rstd the forward saved. */
void orc_rmsnorm_bwd(int64_t T, int64_t H,
                     const uint16_t *g, int64_t ldg,
                     const uint16_t *x, int64_t ldx,
                     const void *w, int w_is_f32, float weight_bias,
                     const float *rstd,
                     const uint16_t *g_res, int64_t ldgr,
                     double *dx_exact, uint16_t *dx, double *m_out,
                     double *dw, double *dw_abs)
{
    double *we = malloc(sizeof(double) * (size_t)H);
    double *gd = malloc(sizeof(double) * (size_t)H);
    double *hd = malloc(sizeof(double) * (size_t)H);
    double *gr = g_res ? malloc(sizeof(double) * (size_t)H) : NULL;
    double *dxv = malloc(sizeof(double) * (size_t)H);
    double *dwr = malloc(sizeof(double) * (size_t)H);
    orc_weight_eff(H, w, w_is_f32, weight_bias, we);
    if (dw)
        memset(dw, 0, sizeof(double) * (size_t)H);
    if (dw_abs)
        memset(dw_abs, 0, sizeof(double) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < H; ++j) {
            gd[j] = orc_bf16_to_f64(g[t * ldg + j]);
            hd[j] = orc_bf16_to_f64(x[t * ldx + j]);
            if (gr)
                gr[j] = orc_bf16_to_f64(g_res[t * ldgr + j]);
        }
        double m = orc_row_bwd_f64(H, gd, hd, we, (double)rstd[t], gr, dxv, dwr);
        if (m_out)
            m_out[t] = m;
        for (int64_t j = 0; j < H; ++j) {
            if (dx_exact)
                dx_exact[t * H + j] = dxv[j];
            if (dx)
                dx[t * H + j] = orc_bf16_from_f64(dxv[j]);
            if (dw)
                dw[j] += dwr[j];
            if (dw_abs)
                dw_abs[j] += fabs(dwr[j]);
        }
    }
    free(we);
    free(gd);
    free(hd);
    free(gr);
    free(dxv);
    free(dwr);
}

/* [API] rmsnorm_quant / fused_add_rmsnorm_quant, [GUIDE] 3.2: the normalised
 * value is converted to FP8 with a static FP32 scale of shape (1,); the scale
 * divides the value before the cast, as [GUIDE] 4 states for layernorm_quant.
 * The FP8 decision is taken on the FP32 value f32(yv / scale). */
void orc_rmsnorm_quant(int64_t T, int64_t H,
                       const uint16_t *x, int64_t ldx,
                       const uint16_t *residual, int64_t ldr,
                       const void *w, int w_is_f32, float weight_bias,
                       float scale, float eps, int fp8_kind,
                       uint16_t *h_new, double *v_exact, uint8_t *q,
                       float *rstd32)
{
    double *h = malloc(sizeof(double) * (size_t)H);
    double *we = malloc(sizeof(double) * (size_t)H);
    double *yv = malloc(sizeof(double) * (size_t)H);
    orc_weight_eff(H, w, w_is_f32, weight_bias, we);
    for (int64_t t = 0; t < T; ++t) {
        load_row(t, H, x, ldx, residual, ldr, h, h_new);
        double r = orc_row_fwd_f64(H, h, we, (double)eps, yv);
        for (int64_t j = 0; j < H; ++j) {
            double v = yv[j] / (double)scale;
            if (v_exact)
                v_exact[t * H + j] = v;
            float v32 = (float)v;
            q[t * H + j] = fp8_kind ? orc_e5m2_from_f32(v32) : orc_e4m3_from_f32(v32);
        }
        if (rstd32)
            rstd32[t] = (float)r;
    }
    free(h);
    free(we);
    free(yv);
}

/* [API] fused_add_rmsnorm_fp8_block_quant, [GUIDE] 3.3: residual = input +
 * residual in place; normed = RMSNorm(residual) * weight stored as BF16;
 * out, block_scale = 1x128 FP8 quantisation of normed with one dynamic FP32
 * scale per row and 128-column block, amax / 448 (448 = largest E4M3FN value),
 * stored column-major as block_scale[b][t] with leading dimension
 * round_up(T, 4). */
void orc_fused_add_rmsnorm_fp8_block_quant(int64_t T, int64_t H,
                       const uint16_t *x, int64_t ldx,
                       const uint16_t *residual, int64_t ldr,
                       const uint16_t *w, float eps,
                       uint16_t *h_new, double *normed_exact, uint16_t *normed,
                       float *block_scale, int64_t ldT, uint8_t *q)
{
    double *h = malloc(sizeof(double) * (size_t)H);
    double *we = malloc(sizeof(double) * (size_t)H);
    double *yv = malloc(sizeof(double) * (size_t)H);
    double *nd = malloc(sizeof(double) * (size_t)H);
    orc_weight_eff(H, w, 0, 0.0f, we);
    for (int64_t t = 0; t < T; ++t) {
        load_row(t, H, x, ldx, residual, ldr, h, h_new);
        (void)orc_row_fwd_f64(H, h, we, (double)eps, yv);
        for (int64_t j = 0; j < H; ++j) {
            uint16_t nb = orc_bf16_from_f64(yv[j]);
            if (normed_exact)
                normed_exact[t * H + j] = yv[j];
            normed[t * H + j] = nb;
            nd[j] = orc_bf16_to_f64(nb);
        }
        for (int64_t b = 0; b < H / 128; ++b) {
            double amax = 0.0;
            for (int64_t j = b * 128; j < b * 128 + 128; ++j)
                if (fabs(nd[j]) > amax)
                    amax = fabs(nd[j]);
            float s = (float)(amax / 448.0);
            block_scale[b * ldT + t] = s;
            for (int64_t j = b * 128; j < b * 128 + 128; ++j)
                q[t * H + j] = (s > 0.0f) ? orc_e4m3_from_f32((float)(nd[j] / (double)s))
                                          : (uint8_t)0;
        }
    }
    free(h);
    free(we);
    free(yv);
    free(nd);
}

/* [ADA] overview: AdaRMSNorm = RMSNorm(x, weight) * (1 + style_scale) +
 * style_shift; Tensor Conventions: style is (rows, 3*dim) or (1, 3*dim)
 * broadcast to every row, its thirds being scale, shift and the gate output. */
void orc_ada_rms_norm_style(int64_t T, int64_t D,
                            const uint16_t *x, const uint16_t *w,
                            const uint16_t *style, int64_t style_rows, float eps,
                            double *out_exact, uint16_t *out, uint16_t *gate_out)
{
    double *h = malloc(sizeof(double) * (size_t)D);
    double *we = malloc(sizeof(double) * (size_t)D);
    double *yv = malloc(sizeof(double) * (size_t)D);
    orc_weight_eff(D, w, 0, 0.0f, we);
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *st = style + (style_rows == 1 ? 0 : t) * 3 * D;
        load_row(t, D, x, D, NULL, 0, h, NULL);
        (void)orc_row_fwd_f64(D, h, we, (double)eps, yv);
        for (int64_t j = 0; j < D; ++j) {
            double sc = orc_bf16_to_f64(st[j]);
            double sh = orc_bf16_to_f64(st[D + j]);
            double ov = yv[j] * (1.0 + sc) + sh;
            if (out_exact)
                out_exact[t * D + j] = ov;
            out[t * D + j] = orc_bf16_from_f64(ov);
            gate_out[t * D + j] = st[2 * D + j];
        }
    }
    free(h);
    free(we);
    free(yv);
}

/* [ADA] overview, fused gate path: residual += x * gate, then AdaRMSNorm of
 * the updated residual, then static FP8.  The update follows BF16 tensor
 * arithmetic: the product x*gate is stored as BF16 and the sum rounded to BF16
 * ([ADA] Validation: residual outputs are bit-exact).  The static scale
 * divides before the E4M3FN cast, decided on the FP32 value. */
void orc_gate_residual_ada_norm_fp8(int64_t T, int64_t D,
                            const uint16_t *residual, const uint16_t *x,
                            const uint16_t *gate, const uint16_t *w,
                            const uint16_t *style, int64_t style_rows,
                            float scale, float eps,
                            uint16_t *residual_out, double *v_exact, uint8_t *q,
                            uint16_t *gate_out)
{
    double *h = malloc(sizeof(double) * (size_t)D);
    double *we = malloc(sizeof(double) * (size_t)D);
    double *yv = malloc(sizeof(double) * (size_t)D);
    orc_weight_eff(D, w, 0, 0.0f, we);
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *st = style + (style_rows == 1 ? 0 : t) * 3 * D;
        for (int64_t j = 0; j < D; ++j) {
            double xg = orc_bf16_to_f64(x[t * D + j]) * orc_bf16_to_f64(gate[t * D + j]);
            double prod = orc_bf16_to_f64(orc_bf16_from_f64(xg));
            uint16_t hn = orc_bf16_from_f64(orc_bf16_to_f64(residual[t * D + j]) + prod);
            residual_out[t * D + j] = hn;
            h[j] = orc_bf16_to_f64(hn);
        }
        (void)orc_row_fwd_f64(D, h, we, (double)eps, yv);
        for (int64_t j = 0; j < D; ++j) {
            double sc = orc_bf16_to_f64(st[j]);
            double sh = orc_bf16_to_f64(st[D + j]);
            double v = (yv[j] * (1.0 + sc) + sh) / (double)scale;
            if (v_exact)
                v_exact[t * D + j] = v;
            q[t * D + j] = orc_e4m3_from_f32((float)v);
            gate_out[t * D + j] = st[2 * D + j];
        }
    }
    free(h);
    free(we);
    free(yv);
}

/* [API] fused_rmsnorm_silu, [GUIDE] 5.1: out = SiLU(RMSNorm(input, weight,
 * eps)) with SiLU(v) = v / (1 + exp(-v)), applied to the unrounded
 * normalised value yv.  BF16 output: bf16(SiLU(yv)).  FP8 output (E4M3FN):
 * the nearest code of the FP32 value f32(SiLU(yv) / scale); the guide names
 * no scale for this operation, so scale = 1 is the plain cast.  v_exact
 * (nullable) receives SiLU(yv) / scale (scale 1 for the BF16 output). */
void orc_fused_rmsnorm_silu(int64_t T, int64_t H,
                            const uint16_t *x, int64_t ldx,
                            const void *w, int w_is_f32, float weight_bias,
                            float eps, int out_fp8, float scale,
                            double *v_exact, uint16_t *y, uint8_t *q,
                            float *rstd32)
{
    double *h = malloc(sizeof(double) * (size_t)H);
    double *we = malloc(sizeof(double) * (size_t)H);
    double *yv = malloc(sizeof(double) * (size_t)H);
    orc_weight_eff(H, w, w_is_f32, weight_bias, we);
    for (int64_t t = 0; t < T; ++t) {
        load_row(t, H, x, ldx, NULL, 0, h, NULL);
        double r = orc_row_fwd_f64(H, h, we, (double)eps, yv);
        for (int64_t j = 0; j < H; ++j) {
            double s = yv[j] / (1.0 + exp(-yv[j]));
            if (out_fp8) {
                double v = s / (double)scale;
                if (v_exact)
                    v_exact[t * H + j] = v;
                q[t * H + j] = orc_e4m3_from_f32((float)v);
            } else {
                if (v_exact)
                    v_exact[t * H + j] = s;
                y[t * H + j] = orc_bf16_from_f64(s);
            }
        }
        if (rstd32)
            rstd32[t] = (float)r;
    }
    free(h);
    free(we);
    free(yv);
}

/* [API] layernorm / layernorm_quant, [GUIDE] 4: BF16 input, FP32 gamma and
 * beta,
 *   out = ((x - E[x]) / sqrt(Var[x] + eps)) * gamma + beta,
 * Var the mean of the squared deviations from E[x] (divisor H: the reading
 * of a layer's variance over its features).  BF16 output: bf16(out).
 * layernorm_quant divides by the FP32 scale before the FP8 cast (E4M3FN or
 * E5M2 by fp8_kind), decided on the FP32 value f32(out / scale).  v_exact
 * (nullable) receives out (BF16) or out / scale (FP8); mean_out and
 * rstd_out (nullable) E[x] and 1 / sqrt(Var[x] + eps) per row. */
void orc_layernorm(int64_t T, int64_t H,
                   const uint16_t *x, int64_t ldx,
                   const float *gamma, const float *beta, float eps,
                   int out_fp8, int fp8_kind, float scale,
                   double *v_exact, uint16_t *y, uint8_t *q,
                   double *mean_out, double *rstd_out)
{
    double *h = malloc(sizeof(double) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        double sum = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            h[j] = orc_bf16_to_f64(x[t * ldx + j]);
            sum += h[j];
        }
        double mean = sum / (double)H;
        double sq = 0.0;
        for (int64_t j = 0; j < H; ++j)
            sq += (h[j] - mean) * (h[j] - mean);
        double var = sq / (double)H;
        double rstd = 1.0 / sqrt(var + (double)eps);
        if (mean_out)
            mean_out[t] = mean;
        if (rstd_out)
            rstd_out[t] = rstd;
        for (int64_t j = 0; j < H; ++j) {
            double o = (h[j] - mean) * rstd * (double)gamma[j] + (double)beta[j];
            if (out_fp8) {
                double v = o / (double)scale;
                if (v_exact)
                    v_exact[t * H + j] = v;
                float v32 = (float)v;
                q[t * H + j] = fp8_kind ? orc_e5m2_from_f32(v32) : orc_e4m3_from_f32(v32);
            } else {
                if (v_exact)
                    v_exact[t * H + j] = o;
                y[t * H + j] = orc_bf16_from_f64(o);
            }
        }
    }
    free(h);
}
