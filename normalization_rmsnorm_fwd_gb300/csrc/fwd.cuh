// fwd.cuh -- the RMSNorm forward row kernel and its epilogues.
//
// One row is owned by a group of `tpr` threads; each thread holds VPT
// vectors of VEC BF16 elements, vector v = k*tpr + lane, so every load and
// store instruction of a group covers a contiguous span of the row.  The
// whole row stays in registers as packed BF16 (the normalised input is BF16
// by definition: x itself, or h_new = bf16(x + residual)), so nothing is
// staged or re-read.  A CTA holds `rpc` row groups.  Groups of <= 32 threads
// (SUB) reduce with warp shuffles only; wider groups add one shared-memory
// step across their warps.
//
// Per row (sources: "FlashInfer normalization operator guide" 2.1-2.4,
// 3.1-3.3, 6.1; "cake_rmsnorm_det_train_forward" Parameters/Returns;
// "flashrt-adaptive-norms" README formula block):
//   h      = x | bf16(x + residual) | bf16(residual + bf16(x * gate))
//   ss     = sum h^2 (FP32 per thread, compensated pairs across threads)
//   (elementwise FP32 arithmetic in packed FP32x2 instructions)
//   rstd   = 1 / sqrt(ss / H + eps)        (IEEE sqrt and division)
//   o      = (h * rstd) * f32(w + bias)
//   then one of the epilogues below.
// LayerNorm rows ("FlashInfer normalization operator guide" 4) take the mean
// first and then the sum of squared deviations from it (plain FP32 sums in a
// fixed tree: the deviations' squares are all positive, and the mean's
// absolute error stays near 2^-21 of mean|x|): rstd = 1 / sqrt(ss_dev / H +
// eps), o = (h - mean)*rstd*gamma + beta.
//
// Two launch forms.  One row per group per CTA (LOOP = false): a grid of
// ceil(T / rpc) CTAs.  Persistent (LOOP = true: the plain row with the y or
// static FP8 epilogue, and LayerNorm with gamma and beta in shared memory;
// each streams a single input): a grid of resident CTAs whose groups walk the
// rows with a stride of the whole grid; the weights are loaded once per CTA
// and the next row's x is fetched ahead (into registers, or into L2 only) so
// its loads are in flight while the current row is reduced and written.
// Every grid is launched with programmatic dependent launch and waits for
// the preceding grid before touching global memory.
#pragma once

#include <atomic>

#include "launch.h"

namespace crmsn {

// Four (two) FP32 values to / from 16-byte (8-byte) aligned shared memory.
// Plain loads, which the compiler may schedule early (measured: faster than
// keeping them in program order with the epilogue's stores).
__device__ __forceinline__ void ld_smem_f32x4(const float *p, float *f)
{
    if (!dbg_shared(p, 16)) { f[0] = f[1] = f[2] = f[3] = 0.f; return; }
    const float4 v = *reinterpret_cast<const float4 *>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void ld_smem_f32x2(const float *p, float *f)
{
    if (!dbg_shared(p, 8)) { f[0] = f[1] = 0.f; return; }
    const float2 v = *reinterpret_cast<const float2 *>(p);
    f[0] = v.x; f[1] = v.y;
}
__device__ __forceinline__ void st_smem_f32x4(float *p, const float *f)
{
    if (!dbg_shared(p, 16)) return;
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
}
__device__ __forceinline__ void st_smem_f32x2(float *p, float a, float b)
{
    if (!dbg_shared(p, 8)) return;
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// SiLU of a pair, v / (1 + exp(-v)), as v * RCP(1 + 2^(-v * log2 e)): the
// products and the sum packed, the base-2 exponential and the reciprocal
// from the approximate hardware instructions (ex2.approx, rcp.approx).  The
// relative error stays near 2^-20 (most of it from rounding v * log2 e, up
// to |v| * 2^-24) -- far below a BF16 half-ulp.  Extremes: for v > ~88 the
// exponential flushes to 0 and the result is v; for v < ~-87 it exceeds
// 2^126, the reciprocal flushes to 0 and the result is -0 (|SiLU(v)| is
// below 1e-35 there); +-inf and NaN give what v * sigmoid(v) gives.
__device__ __forceinline__ F2 silu_f2(F2 v)
{
    const F2 t = f2_mul(v, f2(-1.4426950408889634f));      // -v * log2(e)
    const F2 d = f2_add(f2(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t))), f2(1.f));
    return f2_mul(v, f2(rcp_approx(f2_lo(d)), rcp_approx(f2_hi(d))));
}

// How the persistent form fetches the next row ahead: 1 = prefetched into
// L2, 2 = loaded into registers (measured per epilogue: the broadcast Ada
// form 9.7 against 10.2 us with 2; the y form 51.6 against 55.7 us with 1;
// LayerNorm with 64 elements per thread, BF16 out, T = 16384, H = 4096:
// 46.5 against 53.0 us with 1).
constexpr int fwd_prefetch(int in, int out, int vpt)
{
    if (in == IN_LAYERNORM) return vpt <= 4 ? 2 : 1;
    return out == OUT_Q || out == OUT_ADA ? 2 : 1;
}

// The kernel body.  WK is the weight kind (WK_MIX: BF16 weight, no bias,
// kept packed and multiplied by h exactly with the mixed-precision FMA;
// WK_BF16 / WK_F32: the effective weight f32(w + bias) in FP32 registers).
template <int IN, int WK, int OUT, int FP8K, int VEC, int VPT, bool SUB, bool LOOP>
__device__ __forceinline__ void fwd_body(const FwdParams &p)
{
    constexpr int NW = VEC / 2;
    constexpr bool ADA = (OUT == OUT_ADA || OUT == OUT_ADA_Q);
    constexpr bool LN = (IN == IN_LAYERNORM);
    constexpr bool WMIX = (WK == WK_MIX) && !LN;
    // Per-warp partial sums of a multi-warp row group.  The persistent form
    // alternates two planes by row parity: the warps of a group write row
    // i+1's slots while slower warps may still read row i's, and only the
    // barrier of row i+1 orders those writes after row i's reads, so row
    // i+2 can reuse plane i's slots.  LayerNorm's two reductions per row
    // use red2_h and then red_h[0], a barrier between every reuse.
    __shared__ float red_h[2][32];
    __shared__ float red2_h[LN ? 32 : 1];
    // Programmatic dependent launch: wait for the preceding grid (and its
    // memory) before any global access; let the next grid be scheduled now
    // (it waits for this whole grid the same way).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    CRMSN_DEBUG_ENTER(p.dbg);

    const int tpr = p.tpr;
    const int grp = row_group(tpr, p.rpc);
    const int lane = threadIdx.x - grp * tpr;
    const int nvec = p.H / VEC;

    // ---------------- phase 1: loads ---------------------------------------
    // Weights: row-independent, in registers (packed BF16 for WK_MIX, else
    // the FP32 effective weight).  LayerNorm's gamma and beta do not stay in
    // registers through its two reductions: the persistent form keeps them
    // in shared memory (loaded once per CTA), the one-row form loads them in
    // its epilogue, vector by vector.
    constexpr bool LN_SMEM = LN && LOOP;
    constexpr bool LN_LATE = LN && !LOOP;
    // The persistent AdaRMSNorm form (a broadcast style row) keeps 1 + scale
    // and shift as FP32 in shared memory (converted once per CTA, the same
    // bits as per row) and the gate chunk of its columns in registers.
    constexpr bool ADA_SMEM = ADA && LOOP;
    // LN_SMEM / ADA_SMEM table: gamma then beta (1 + scale then shift), 2H
    // floats; for 16-byte vectors each stored as two planes (the first and
    // the last four values of every vector), so that a warp's 16-byte reads
    // of consecutive vectors hit distinct banks.
    extern __shared__ __align__(16) unsigned char fwd_dyn_smem[];
    float *const ln_gb = reinterpret_cast<float *>(fwd_dyn_smem);
    BVec<VEC> wb[VPT];
    float wf[VPT][VEC], bt[VPT][VEC];
    auto load_weight_vec = [&](int k) {
        if constexpr (LN) return;
        const int v = k * tpr + lane;
        if (v < nvec) {
            const int64_t c = (int64_t)v * VEC;
            if constexpr (WK == WK_F32) {
                ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, wf[k]);
#pragma unroll
                for (int i = 0; i < VEC; ++i) wf[k][i] = __fadd_rn(wf[k][i], p.bias);
            } else if constexpr (WK == WK_BF16) {
                const BVec<VEC> b = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    wf[k][2 * i] = __fadd_rn(bf_lo(b.w[i]), p.bias);
                    wf[k][2 * i + 1] = __fadd_rn(bf_hi(b.w[i]), p.bias);
                }
            } else {
                wb[k] = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
            }
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i) wb[k].w[i] = 0u;
#pragma unroll
            for (int i = 0; i < VEC; ++i) wf[k][i] = 0.f;
        }
    };
    auto load_weights = [&]() {
#pragma unroll
        for (int k = 0; k < VPT; ++k) load_weight_vec(k);
    };
    // The row's streamed inputs: x (into xs), residual, gate, style, and with
    // `weights` the weight vectors too (interleaved per vector: fewer live
    // registers than all of one tensor first).
    BVec<VEC> xa[VPT], ra[VPT], ga[VPT];
    BVec<VEC> sc[VPT], sh[VPT], gt[VPT];
    auto load_row = [&](int64_t t, BVec<VEC> (&xs)[VPT], bool weights) {
        const bool live = t < p.T;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (weights) load_weight_vec(k);
            const int v = k * tpr + lane;
            if (live && v < nvec) {
                const int64_t c = (int64_t)v * VEC;
                xs[k] = ld_stream<VEC>(p.x + t * p.ldx + c);
                if constexpr (IN == IN_RESIDUAL || IN == IN_GATED)
                    ra[k] = ld_stream<VEC>(p.r + t * p.ldr + c);
                if constexpr (IN == IN_GATED)
                    ga[k] = ld_stream<VEC>(p.gate + t * p.ldgate + c);
                if constexpr (ADA && !ADA_SMEM) {
                    const uint16_t *srow = p.style + t * p.lds;
                    if (p.lds == 0) {
                        sc[k] = ld_keep<VEC>(srow + c);
                        sh[k] = ld_keep<VEC>(srow + p.H + c);
                        gt[k] = ld_keep<VEC>(srow + 2 * p.H + c);
                    } else {
                        sc[k] = ld_stream<VEC>(srow + c);
                        sh[k] = ld_stream<VEC>(srow + p.H + c);
                        gt[k] = ld_stream<VEC>(srow + 2 * p.H + c);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    xs[k].w[i] = 0u; ra[k].w[i] = 0u; ga[k].w[i] = 0u;
                    sc[k].w[i] = 0u; sh[k].w[i] = 0u; gt[k].w[i] = 0u;
                }
            }
        }
    };

    // Phases 2-4 of row t, whose inputs are in xa (and ra, ga, sc, sh, gt).
    // Every thread of the CTA calls it the same number of times (it may
    // contain CTA barriers).
    // The static FP8 scale, read once (after the dependency wait at the top)
    // as its correctly rounded reciprocal: the epilogues multiply by it
    // (for the plain static-scale form folded into rstd), within a few FP32
    // ulps of the quotient v / scale, so a code can differ from the one of
    // the exact quotient only next to a rounding midpoint.
    float inv_scale = 1.f;
    if constexpr (OUT == OUT_Q || OUT == OUT_ADA_Q)
        inv_scale = __frcp_rn(ld_f32_ro(p.scale));
    if constexpr (OUT == OUT_SILU_Q)
        inv_scale = p.scale != nullptr ? __frcp_rn(ld_f32_ro(p.scale)) : 1.f;
    // The static-scale RMSNorm form scales rstd instead of every value.
    constexpr bool FOLD_SCALE = OUT == OUT_Q && !LN;

    // The barrier between a multi-warp group's per-warp slots and their
    // readers.  LayerNorm and SiLU use the group's own named barrier (1 +
    // group, the group's threads) when the CTA holds several groups, so that
    // one group's row does not wait for another's (measured: LayerNorm 3 %,
    // SiLU 2 % faster); the other forms keep the CTA barrier, since a kernel
    // with a named barrier of a run-time id reserves all 16 barriers and ran
    // 1-5 % slower there.
    constexpr bool GROUP_BAR = LN || OUT == OUT_SILU || OUT == OUT_SILU_Q;
    auto group_sync = [&]() {
        if (GROUP_BAR && p.rpc > 1)
            asm volatile("bar.sync %0, %1;" :: "r"(1 + grp), "r"(tpr) : "memory");
        else
            __syncthreads();
    };

    // Sum over the row group of one FP32 value per thread, in plain FP32 and
    // a fixed order: a butterfly within each warp (within the group for
    // groups of <= 32 threads), then, across the group's warps, every warp
    // adds the group's per-warp slots in the same butterfly.  Every thread
    // of the group gets the same bits.  (The statistics are sums of
    // non-negative squares, or LayerNorm's mean and squared deviations; a
    // fixed FP32 tree keeps rstd within a few FP32 ulps.)
    auto row_sum = [&](float v, float *rh) -> float {
        const int width = SUB ? tpr : 32;
        for (int o = width >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if constexpr (!SUB) {
            const int nwarp = tpr >> 5;
            const int warp = threadIdx.x >> 5;
            if ((threadIdx.x & 31) == 0) rh[warp] = v;
            group_sync();
            int w = 1;
            while (w < nwarp) w <<= 1;
            const int i = threadIdx.x & (w - 1);
            v = i < nwarp ? rh[grp * nwarp + i] : 0.f;
            for (int o = w >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        }
        return v;
    };

    // The two halves of row_sum for a multi-warp group, with the CTA barrier
    // between them left to the caller (the pipelined persistent loop).
    auto publish = [&](float v, float *rh) {
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if ((threadIdx.x & 31) == 0) rh[threadIdx.x >> 5] = v;
    };
    auto gather = [&](const float *rh) -> float {
        const int nwarp = tpr >> 5;
        int w = 1;
        while (w < nwarp) w <<= 1;
        const int i = threadIdx.x & (w - 1);
        float v = i < nwarp ? rh[grp * nwarp + i] : 0.f;
        for (int o = w >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        return v;
    };

    // Phase 2 of row t from the loaded words: the normalised input h into
    // hh (h_new stored on the residual routes) and this thread's partial sum
    // (of h^2, or of h for LayerNorm).
    auto phase_h = [&](int64_t t, BVec<VEC> (&h)[VPT]) -> float {
        const bool live = t < p.T;
        // Four independent chains: the sum of squares (RMSNorm) or of h
        // (LayerNorm's mean).
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                const uint32_t xw = xa[k].w[i];
                uint32_t hw;
                if constexpr (IN == IN_PLAIN || LN) {
                    hw = xw;
                } else if constexpr (IN == IN_RESIDUAL) {
                    // The FP32 sum of two BF16 values rounded once to BF16 is the
                    // correctly rounded BF16 sum (double rounding is innocuous).
                    hw = bf16_f2(f2_add(f2_bf16(xw), f2_bf16(ra[k].w[i])));
                } else {
                    // bf16(x * gate) first (the FP32 product of two BF16 values is
                    // exact), then the BF16 residual add.
                    const uint32_t pw = bf16_f2(mul_bf16x2(xw, ga[k].w[i]));
                    hw = bf16_f2(f2_add(f2_bf16(ra[k].w[i]), f2_bf16(pw)));
                }
                h[k].w[i] = hw;
                const int j = (k * NW + i) & 1;
                if constexpr (LN)
                    acc_bf16x2(hw, acc[2 * j], acc[2 * j + 1]);     // sum of h (the mean first)
                else
                    sq_acc_bf16x2(hw, acc[2 * j], acc[2 * j + 1]);  // h^2 exact, one rounding each
            }
            if constexpr (IN != IN_PLAIN && !LN) {
                const int v = k * tpr + lane;
                if (live && v < nvec)
                    st_stream<VEC>(p.hn + t * p.ldh + (int64_t)v * VEC, h[k]);
            }
        }
        return __fadd_rn(__fadd_rn(acc[0], acc[2]), __fadd_rn(acc[1], acc[3]));
    };

    // LayerNorm: this thread's sum of squared deviations from the mean (none
    // past the row), h - mean formed from the BF16 halves directly.
    auto dev_part = [&](int64_t t, const BVec<VEC> (&h)[VPT], float mean) -> float {
        const bool live = t < p.T;
        F2 ss2 = f2(0.f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const bool ok = live && k * tpr + lane < nvec;
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                const F2 d = add_bf16x2(h[k].w[i], -mean);
                if (ok) ss2 = f2_fma(d, d, ss2);
            }
        }
        return __fadd_rn(f2_lo(ss2), f2_hi(ss2));
    };

    // Phases 3-4 of row t from h and its partial sum: the row reduction, rstd,
    // the epilogue.  With `reduced` (RMSNorm only) the pipelined loop has
    // reduced the row already and `part` is the total.
    auto finish = [&](int64_t t, BVec<VEC> (&h)[VPT], float part, int par, bool reduced) {
        const bool live = t < p.T;
        // ---------------- phase 3: row reduction -> rstd ----------------------
        // The row's FP32 values are unpacked again from the BF16 words after
        // each reduction instead of being kept (twice the registers) across
        // it: the empty asm makes the words opaque to the compiler.  Measured
        // per variant: it pays where the epilogue is long (SiLU, block
        // quantisation, one-row LayerNorm) and in the persistent y form.
        constexpr bool REUNPACK = (LN && !LOOP) || OUT == OUT_SILU || OUT == OUT_SILU_Q ||
                                  OUT == OUT_BLOCK || (LOOP && OUT == OUT_Y && !LN);
        auto reunpack = [&]() {
            if constexpr (REUNPACK) {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int i = 0; i < NW; ++i) asm volatile("" : "+r"(h[k].w[i]));
            }
        };
        float mean = 0.f;
        float ssum;
        if constexpr (LN) {
            mean = __fdiv_rn(row_sum(part, red2_h), (float)p.H);
            reunpack();
            ssum = row_sum(dev_part(t, h, mean), red_h[0]);
            if (p.mean != nullptr && live && lane == 0)
                st_f32(p.mean + t, mean);
        } else {
            ssum = reduced ? part : row_sum(part, red_h[par]);
        }
        reunpack();
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ssum, (float)p.H), p.eps)));
        if (p.rstd != nullptr && live && lane == 0)
            st_f32(p.rstd + t, rstd);

        // ---------------- phase 4: epilogue -----------------------------------
        // o = (h * w) * rstd with h * w exact (WK_MIX), or (h * rstd) * w_eff;
        // for the static FP8 form rstd carries the reciprocal scale.
        // The fold needs rstd / scale to be a normal FP32 number (a tiny scale
        // and an eps-sized row can overflow it); otherwise each value is scaled.
        const float rq = __fmul_rn(rstd, inv_scale);
        const bool folded = FOLD_SCALE && fabsf(rq) <= 0x1.fffffep127f && fabsf(rq) >= 0x1p-126f;
        const F2 rstd2 = f2(folded ? rq : rstd);
        const F2 inv2 = f2(inv_scale);

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            const bool ok = live && v < nvec;
            const int64_t c = (int64_t)v * VEC;
            if constexpr (LN_SMEM || ADA_SMEM) {
                if (v < nvec) {
                    if constexpr (VEC == 8) {
                        const int hp = p.H >> 1;
                        ld_smem_f32x4(ln_gb + v * 4, wf[k]);
                        ld_smem_f32x4(ln_gb + hp + v * 4, wf[k] + 4);
                        ld_smem_f32x4(ln_gb + p.H + v * 4, bt[k]);
                        ld_smem_f32x4(ln_gb + p.H + hp + v * 4, bt[k] + 4);
                    } else {
                        ld_smem_f32x2(ln_gb + c, wf[k]);
                        ld_smem_f32x2(ln_gb + p.H + c, bt[k]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) { wf[k][i] = 0.f; bt[k][i] = 0.f; }
                }
            }
            if constexpr (LN_LATE) {
                if (v < nvec) {
                    ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, wf[k]);
                    ld_f32_keep<VEC>(p.beta + c, bt[k]);
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) { wf[k][i] = 0.f; bt[k][i] = 0.f; }
                }
            }
            F2 o[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                if constexpr (LN)
                    o[i] = f2_fma(f2_mul(add_bf16x2(h[k].w[i], -mean), rstd2),
                                  f2(wf[k][2 * i], wf[k][2 * i + 1]), f2(bt[k][2 * i], bt[k][2 * i + 1]));
                else if constexpr (WMIX)
                    o[i] = f2_mul(mul_bf16x2(h[k].w[i], wb[k].w[i]), rstd2);
                else
                    o[i] = f2_mul(f2_mul(f2_bf16(h[k].w[i]), rstd2), f2(wf[k][2 * i], wf[k][2 * i + 1]));
            }

            if constexpr (OUT == OUT_Y) {
                BVec<VEC> yv;
#pragma unroll
                for (int i = 0; i < NW; ++i) yv.w[i] = bf16_f2(o[i]);
                if (ok) st_stream<VEC>(p.y + t * p.ldy + c, yv);
            } else if constexpr (OUT == OUT_Q) {
                uint32_t cq[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    const F2 v = folded ? o[i] : f2_mul(o[i], inv2);
                    cq[i] = pack_fp8<FP8K>(f2_lo(v), f2_hi(v));
                }
                if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
            } else if constexpr (OUT == OUT_BLOCK) {
                // normed = bf16(o); amax over the 128-column block held by 16
                // consecutive lanes (VEC == 8, tpr a multiple of 16).
                BVec<VEC> nv;
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    nv.w[i] = bf16_f2(o[i]);
                    amax = fmaxf(amax, fmaxf(fabsf(bf_lo(nv.w[i])), fabsf(bf_hi(nv.w[i]))));
                }
                if (ok) st_stream<VEC>(p.y + t * p.ldy + c, nv);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                const float s = __fdiv_rn(amax, 448.0f);
                const DivScale bdiv(s);
                uint32_t cq[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    if (s > 0.f) {
                        float a, b;
                        bdiv.div(f2_bf16(nv.w[i]), a, b);
                        cq[i] = pack_fp8<0>(a, b);
                    } else {
                        cq[i] = 0u;
                    }
                }
                if (ok) {
                    st_fp8<VEC>(p.q + t * p.ldq + c, cq);
                    if ((v & 15) == 0)
                        st_f32(p.bscale + (int64_t)(v >> 4) * p.ldT + t, s);
                }
            } else if constexpr (OUT == OUT_SILU) {
                BVec<VEC> yv;
#pragma unroll
                for (int i = 0; i < NW; ++i) yv.w[i] = bf16_f2(silu_f2(o[i]));
                if (ok) st_stream<VEC>(p.y + t * p.ldy + c, yv);
            } else if constexpr (OUT == OUT_SILU_Q) {
                uint32_t cq[NW];
                if (p.scale == nullptr) {      // the plain cast (no division by 1)
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        const F2 y2 = silu_f2(o[i]);
                        cq[i] = pack_fp8<0>(f2_lo(y2), f2_hi(y2));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        const F2 y2 = f2_mul(silu_f2(o[i]), inv2);
                        cq[i] = pack_fp8<0>(f2_lo(y2), f2_hi(y2));
                    }
                }
                if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
            } else {  // ADA: o * (1 + scale) + shift, one FP32 rounding (fma)
                const F2 one2 = f2(1.f);
                F2 ov[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    if constexpr (ADA_SMEM)
                        ov[i] = f2_fma(o[i], f2(wf[k][2 * i], wf[k][2 * i + 1]), f2(bt[k][2 * i], bt[k][2 * i + 1]));
                    else
                        ov[i] = f2_fma(o[i], f2_add(one2, f2_bf16(sc[k].w[i])), f2_bf16(sh[k].w[i]));
                }
                if constexpr (OUT == OUT_ADA) {
                    BVec<VEC> out;
#pragma unroll
                    for (int i = 0; i < NW; ++i) out.w[i] = bf16_f2(ov[i]);
                    if (ok) st_stream<VEC>(p.y + t * p.ldy + c, out);
                } else {
                    uint32_t cq[NW];
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        const F2 v = f2_mul(ov[i], inv2);
                        cq[i] = pack_fp8<0>(f2_lo(v), f2_hi(v));
                    }
                    if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
                }
                if (ok) st_stream<VEC>(p.gate_out + t * p.ldgo + c, gt[k]);
            }
        }
    };

    auto process = [&](int64_t t, int par) {
        BVec<VEC> h[VPT];
        const float part = phase_h(t, h);
        finish(t, h, part, par, false);
    };

    if constexpr (!LOOP) {
        const int64_t t = (int64_t)blockIdx.x * p.rpc + grp;
        load_row(t, xa, true);
        process(t, 0);
    } else {
        static_assert(IN == IN_PLAIN || LN || ADA, "no persistent form for this input");
        load_weights();
        const int64_t stride = (int64_t)gridDim.x * p.rpc;
        const int64_t b0 = (int64_t)blockIdx.x * p.rpc;
        constexpr int PF = fwd_prefetch(IN, OUT, VPT);
        load_row(b0 + grp, xa, false);
        if constexpr (LN_SMEM) {
            // gamma and beta into shared memory, the whole CTA striding over
            // the vectors (the first row's loads are already in flight).
            const float *gam = static_cast<const float *>(p.w);
            for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
                float g[VEC], b[VEC];
                ld_f32_keep<VEC>(gam + (int64_t)v * VEC, g);
                ld_f32_keep<VEC>(p.beta + (int64_t)v * VEC, b);
                if constexpr (VEC == 8) {
                    const int hp = p.H >> 1;
                    st_smem_f32x4(ln_gb + v * 4, g);
                    st_smem_f32x4(ln_gb + hp + v * 4, g + 4);
                    st_smem_f32x4(ln_gb + p.H + v * 4, b);
                    st_smem_f32x4(ln_gb + p.H + hp + v * 4, b + 4);
                } else {
                    st_smem_f32x2(ln_gb + v * 2, g[0], g[1]);
                    st_smem_f32x2(ln_gb + p.H + v * 2, b[0], b[1]);
                }
            }
            __syncthreads();
        }
        if constexpr (ADA_SMEM) {
            // 1 + scale and shift of the broadcast style row into shared
            // memory (the whole CTA striding over the vectors); the gate
            // chunk of this thread's columns into registers.
            for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
                const int64_t c = (int64_t)v * VEC;
                const BVec<VEC> a = ld_keep<VEC>(p.style + c);
                const BVec<VEC> b = ld_keep<VEC>(p.style + p.H + c);
                float g[VEC], f[VEC];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    const F2 s1 = f2_add(f2(1.f), f2_bf16(a.w[i]));
                    const F2 sf = f2_bf16(b.w[i]);
                    g[2 * i] = f2_lo(s1); g[2 * i + 1] = f2_hi(s1);
                    f[2 * i] = f2_lo(sf); f[2 * i + 1] = f2_hi(sf);
                }
                if constexpr (VEC == 8) {
                    const int hp = p.H >> 1;
                    st_smem_f32x4(ln_gb + v * 4, g);
                    st_smem_f32x4(ln_gb + hp + v * 4, g + 4);
                    st_smem_f32x4(ln_gb + p.H + v * 4, f);
                    st_smem_f32x4(ln_gb + p.H + hp + v * 4, f + 4);
                } else {
                    st_smem_f32x2(ln_gb + v * 2, g[0], g[1]);
                    st_smem_f32x2(ln_gb + p.H + v * 2, f[0], f[1]);
                }
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * tpr + lane;
                if (v < nvec) {
                    gt[k] = ld_keep<VEC>(p.style + 2 * p.H + (int64_t)v * VEC);
                } else {
#pragma unroll
                    for (int i = 0; i < NW; ++i) gt[k].w[i] = 0u;
                }
            }
            __syncthreads();
        }
        // The next row is loaded into registers before this row is processed
        // (PF == 2), or only prefetched into L2 then and loaded afterwards
        // (PF == 1: no registers held across the row).
        auto prefetch_l2 = [&](int64_t t) {
            if (t < p.T) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * tpr + lane;
                    if (v < nvec) {
                        const int64_t c = (int64_t)v * VEC;
                        asm volatile("prefetch.global.L2 [%0];" :: "l"(p.x + t * p.ldx + c));
                        if constexpr (IN == IN_GATED) {
                            asm volatile("prefetch.global.L2 [%0];" :: "l"(p.r + t * p.ldr + c));
                            asm volatile("prefetch.global.L2 [%0];" :: "l"(p.gate + t * p.ldgate + c));
                        }
                    }
                }
            }
        };
        // Measured: the row after next pays for the static FP8 form only
        // (38.7 against 40.9 us at T = H = 8192; the y form lost 5 %).
        constexpr bool AHEAD2 = OUT == OUT_Q && !LN;
        // The static FP8 form with multi-warp rows runs a software pipeline
        // with one CTA barrier per row: iteration k adds up row k's total
        // from the per-warp slots published before the barrier, forms row
        // k + 1's h and partial sum and publishes it (the other plane of
        // slots), starts the loads of row k + 2, then writes row k's outputs
        // -- so the reduction's dependent chain overlaps the next row's
        // arithmetic instead of stalling the CTA.  Measured at T = H = 8192:
        // 34.5 against 38.7 us; the y and AdaRMSNorm forms, which hold at
        // most the next row, lost 9-25 % with it,
        // and LayerNorm (three rows in flight, one barrier instead of two per
        // row) lost 19 % at T = 16384, H = 4096.
        constexpr bool PIPED = OUT == OUT_Q && !LN && !SUB;
        if constexpr (PIPED) {
            BVec<VEC> hc[VPT], hn[VPT];
            const int64_t t0 = b0 + grp;
            publish(phase_h(t0, hc), red_h[0]);
            if (b0 + stride < p.T) load_row(t0 + stride, xa, false);
            group_sync();
            int par = 0;
            for (int64_t base = b0; base < p.T; base += stride, par ^= 1) {
                const int64_t t = base + grp;
                const float total = gather(red_h[par]);
                const bool more = base + stride < p.T;   // the same for the whole CTA
                if (more) {
                    publish(phase_h(t + stride, hn), red_h[par ^ 1]);
                    if (base + 2 * stride < p.T) {
                        if constexpr (AHEAD2) prefetch_l2(t + 3 * stride);
                        load_row(t + 2 * stride, xa, false);
                    }
                }
                finish(t, hc, total, par, true);
                if (more) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) hc[k] = hn[k];
                }
                group_sync();
            }
            return;
        }
        int par = 0;
        for (int64_t base = b0; base < p.T; base += stride, par ^= 1) {
            BVec<VEC> xn[VPT];
            const bool more = base + stride < p.T;   // the same for the whole CTA
            const int64_t tn = base + stride + grp;
            if constexpr (PF == 2) {
                if constexpr (AHEAD2) prefetch_l2(tn + stride);
                if (more) load_row(tn, xn, false);
            } else {
                if (more) prefetch_l2(tn);
            }
            process(base + grp, par);
            if (more) {
                if constexpr (PF == 2) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) xa[k] = xn[k];
                } else {
                    load_row(tn, xa, false);
                }
            }
        }
    }
}

// No minimum CTA count in the launch bounds: an explicit one (even 1) lets
// the compiler take far more registers for these kernels.
template <int IN, int WK, int OUT, int FP8K, int VEC, int VPT, bool SUB, bool LOOP>
__global__ void __launch_bounds__(kFwdMaxThreads) k_rmsnorm_fwd(const FwdParams p)
{
    fwd_body<IN, WK, OUT, FP8K, VEC, VPT, SUB, LOOP>(p);
}

// The same body for the one-row y, static-FP8 and block-FP8 forms of the
// widest rows (512-thread row groups, 32 elements per thread): launch
// bounds that ask for two CTAs per SM hold it to 64 registers (measured at
// T = 4096, H = 16384: 81-93 against 91-112 us for the fused residual
// forward, 73-86 against 84-101 us with the static FP8 epilogue, for every
// weight kind; 98 against 126 us with block FP8).  The AdaRMSNorm, SiLU
// and LayerNorm one-row forms gain nothing from it, and the gated FP8 form
// spills (296 against 206 us).
template <int IN, int WK, int OUT, int FP8K, int VEC, int VPT, bool SUB, bool LOOP>
__global__ void __launch_bounds__(512, 2) k_rmsnorm_fwd_wide(const FwdParams p)
{
    fwd_body<IN, WK, OUT, FP8K, VEC, VPT, SUB, LOOP>(p);
}

// Host-side launch of one kernel.  The persistent form runs on at most
// (resident CTAs per SM) x (SMs) CTAs; the residency for a block size and
// shared-memory size is computed once and remembered.
template <int IN, int WK, int OUT, int FP8K, int VEC, int VPT, bool SUB, bool LOOP>
cudaError_t launch_fwd_kernel(const FwdParams &p, size_t smem, cudaStream_t s)
{
    auto kern = k_rmsnorm_fwd<IN, WK, OUT, FP8K, VEC, VPT, SUB, LOOP>;
    const int threads = p.tpr * p.rpc;
    int64_t blocks = (p.T + p.rpc - 1) / p.rpc;
    if (smem > 0) {
        static std::atomic<int> opted[kOptInDevices];
        cudaError_t e = opt_in_smem(kern, smem, opted);
        if (e != cudaSuccess) return e;
    }
    if constexpr (LOOP) {
        // threads << 40 | shared-memory bytes << 8 | CTAs per SM
        static std::atomic<long long> cached{0};
        const long long key = ((long long)threads << 40) | ((long long)smem << 8);
        long long c = cached.load(std::memory_order_relaxed);
        int per_sm = (int)(c & 0xff);
        if ((c & ~0xffLL) != key || per_sm <= 0) {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) return cudaErrorInvalidConfiguration;
            if (per_sm > 255) per_sm = 255;
            cached.store(key | per_sm, std::memory_order_relaxed);
        }
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t cap = (int64_t)per_sm * sms;
        if (blocks > cap) blocks = cap;
    }
    if constexpr (!LOOP && !SUB && VPT == 4 && (OUT == OUT_Y || OUT == OUT_Q || OUT == OUT_BLOCK))
        if (threads == 512)
            return launch_pdl(k_rmsnorm_fwd_wide<IN, WK, OUT, FP8K, VEC, VPT, SUB, LOOP>,
                              dim3((unsigned)blocks), dim3(threads), smem, s, p);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(threads), smem, s, p);
}

// LayerNorm keeps gamma and beta (2H floats) in shared memory in the
// persistent form up to this size; wider rows use the one-row form.
constexpr size_t kLnSmemMax = 64 * 1024;

// Launch of one instantiation.  Measured: the persistent form pays off for
// the plain row with the y and static FP8 epilogues, for LayerNorm with
// gamma and beta in shared memory and for AdaRMSNorm with a broadcast style
// row in shared memory; SiLU (bound by its arithmetic) runs faster in the
// one-row form.
template <int IN, int WK, int OUT, int FP8K, int VEC, int VPT, bool SUB>
cudaError_t launch_fwd_inst(const FwdParams &p, cudaStream_t s)
{
    if constexpr (IN == IN_LAYERNORM) {
        const size_t table = (size_t)2 * p.H * sizeof(float);
        if (table <= kLnSmemMax)
            return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, true>(p, table, s);
        return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, false>(p, 0, s);
    } else if constexpr (OUT == OUT_ADA || OUT == OUT_ADA_Q) {
        // A broadcast style row (lds == 0) for AdaRMSNorm: the persistent
        // form with the style's 1 + scale and shift in shared memory (2H
        // floats; 10.2 against 11.4 us one row per group at 2520 x 3072).
        // The gated FP8 form, with three input streams, runs one row per
        // group either way (15.5 against 16.2 us persistent).
        if constexpr (OUT == OUT_ADA)
            if (p.lds == 0)
                return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, true>(
                    p, (size_t)2 * p.H * sizeof(float), s);
        return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, false>(p, 0, s);
    } else {
        constexpr bool LOOP = IN == IN_PLAIN && (OUT == OUT_Y || OUT == OUT_Q);
        // The plain y form of a packed BF16 weight runs one row per group up
        // to H = 8192 (measured at T*H = 2^26: 0.96-1.00 of the copy peak
        // against 0.85-0.89 persistent; at H = 16384 0.81 against 0.92); an
        // FP32 or biased weight, which the one-row form reloads for every
        // row, and the static FP8 form stay persistent.
        if constexpr (LOOP && OUT == OUT_Y && WK == WK_MIX)
            if (p.H <= 8192) return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, false>(p, 0, s);
        return launch_fwd_kernel<IN, WK, OUT, FP8K, VEC, VPT, SUB, LOOP>(p, 0, s);
    }
}

// Dispatch over the row layouts the host chooser can return: SUB groups with
// VPT 1|2; multi-warp groups with VPT 2|4 (16-byte vectors) or 2|4|8|16
// (4-byte vectors), i.e. at most 32 elements per thread; and LayerNorm with
// BF16 output also VPT 8 of 16-byte vectors (64 elements per thread).
template <int IN, int WK, int OUT, int FP8K, int VEC>
cudaError_t launch_fwd_vec(const FwdParams &p, int vpt, bool sub, cudaStream_t s)
{
    if (sub) {
        if (vpt == 1) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 1, true>(p, s);
        if (vpt == 2) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 2, true>(p, s);
    } else {
        if (vpt == 2) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 2, false>(p, s);
        if (vpt == 4) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 4, false>(p, s);
        if constexpr (VEC == 8 && IN == IN_LAYERNORM && OUT == OUT_Y)
            if (vpt == 8) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 8, false>(p, s);
        if constexpr (VEC == 2) {
            if (vpt == 8) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 8, false>(p, s);
            if (vpt == 16) return launch_fwd_inst<IN, WK, OUT, FP8K, VEC, 16, false>(p, s);
        }
    }
    return cudaErrorInvalidConfiguration;
}

template <int IN, int WK, int OUT, int FP8K>
cudaError_t launch_fwd(const FwdParams &p, int vec, int vpt, bool sub, cudaStream_t s)
{
    if (vec == 8) return launch_fwd_vec<IN, WK, OUT, FP8K, 8>(p, vpt, sub, s);
    if constexpr (OUT != OUT_BLOCK)
        if (vec == 2) return launch_fwd_vec<IN, WK, OUT, FP8K, 2>(p, vpt, sub, s);
    return cudaErrorInvalidConfiguration;
}

}  // namespace crmsn
