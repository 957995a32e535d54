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
// ceil(T / rpc) CTAs.  Persistent (LOOP = true, the plain row with the y or
// static FP8 epilogue, which streams a single input): a grid of resident CTAs
// whose groups walk the rows with a stride of the whole grid; the weights are
// loaded once per CTA and the next row's x is loaded before the current row
// is reduced and written, so its loads are in flight during that work.
#pragma once

#include <atomic>

#include "launch.h"

namespace crmsn {

// SiLU(v) = v / (1 + exp(-v)) as v * sigmoid(v) with e = exp(-|v|) in (0, 1]
// (no overflow for any finite v): sigmoid = 1 / (1 + e) for v >= 0 and
// e / (1 + e) otherwise.  __expf and the approximate reciprocal of 1 + e (in
// [1, 2]) keep the relative error near 2^-20 for |v| < 10 and far below a
// BF16 half-ulp everywhere.
__device__ __forceinline__ float silu_f32(float v)
{
    const float e = __expf(-fabsf(v));
    const float r = __fdividef(1.0f, 1.0f + e);
    return v * (v >= 0.f ? r : e * r);
}

template <int IN, bool W32, int OUT, int FP8K, int VEC, int VPT, bool SUB, bool LOOP>
__global__ void __launch_bounds__(kFwdMaxThreads)
k_rmsnorm_fwd(const FwdParams p)
{
    constexpr int NW = VEC / 2;
    constexpr bool ADA = (OUT == OUT_ADA || OUT == OUT_ADA_Q);
    constexpr bool LN = (IN == IN_LAYERNORM);
    __shared__ float red_h[32], red_l[32];
    __shared__ float red2_h[LN ? 32 : 1];
    // Programmatic dependent launch: wait for the preceding grid (and its
    // memory) before any global access; let the next grid be scheduled now
    // (it waits for this whole grid the same way).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int tpr = p.tpr;
    const int grp = threadIdx.x / tpr;
    const int lane = threadIdx.x - grp * tpr;
    const int nvec = p.H / VEC;

    // ---------------- phase 1: loads ---------------------------------------
    // Weights (and LayerNorm's beta): row-independent.  LayerNorm loads gamma
    // and beta in its epilogue instead, vector by vector, so that they do not
    // hold registers through the two reductions.
    constexpr bool LN_LATE = LN;
    BVec<VEC> wb[VPT];
    float wf[VPT][VEC], bt[VPT][VEC];
    auto load_weight_vec = [&](int k) {
        if constexpr (LN_LATE) return;
        const int v = k * tpr + lane;
        if (v < nvec) {
            const int64_t c = (int64_t)v * VEC;
            if constexpr (W32)
                ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, wf[k]);
            else
                wb[k] = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
            if constexpr (LN) ld_f32_keep<VEC>(p.beta + c, bt[k]);
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i) wb[k].w[i] = 0u;
#pragma unroll
            for (int i = 0; i < VEC; ++i) { wf[k][i] = 0.f; bt[k][i] = 0.f; }
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
                if constexpr (ADA) {
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
    auto process = [&](int64_t t) {
        const bool live = t < p.T;
        // ---------------- phase 2: normalised input h, sum of squares ---------
        BVec<VEC> h[VPT];
        F2 ss2 = f2(0.f);
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
                    const uint32_t pw = bf16_f2(f2_mul(f2_bf16(xw), f2_bf16(ga[k].w[i])));
                    hw = bf16_f2(f2_add(f2_bf16(ra[k].w[i]), f2_bf16(pw)));
                }
                h[k].w[i] = hw;
                const F2 h2 = f2_bf16(hw);
                if constexpr (LN)
                    ss2 = f2_add(h2, ss2);          // sum of h (the mean comes first)
                else
                    ss2 = f2_fma(h2, h2, ss2);      // h^2 is exact in FP32: one rounding
            }
            if constexpr (IN != IN_PLAIN && !LN) {
                const int v = k * tpr + lane;
                if (live && v < nvec)
                    st_stream<VEC>(p.hn + t * p.ldh + (int64_t)v * VEC, h[k]);
            }
        }

        // ---------------- phase 3: row reduction -> rstd ----------------------
        // Compensated sum over the row group of a per-thread FP32 pair: shuffles
        // within a group of <= 32 threads; otherwise a butterfly within each warp,
        // then across the group's warps (short latency for these short-lived CTAs).
        auto row_sum = [&](F2 part, float *rh, float *rl) -> float {
            float sh_, sl_;
            two_sum(f2_lo(part), f2_hi(part), sh_, sl_);
            if constexpr (SUB) {
                pair_reduce_lanes(sh_, sl_, tpr);
            } else {
                pair_reduce_lanes(sh_, sl_, 32);
                const int nwarp = tpr >> 5;
                const int warp = threadIdx.x >> 5;
                if ((threadIdx.x & 31) == 0) {
                    rh[warp] = sh_;
                    rl[warp] = sl_;
                }
                __syncthreads();
                pair_reduce_warps(sh_, sl_, rh, rl, grp * nwarp, nwarp);
            }
            return __fadd_rn(sh_, sl_);
        };
        // The same sum in plain FP32 (a fixed butterfly, then the group's
        // warps in a fixed tree): LayerNorm's two sums, whose accuracy needs
        // are met without compensation.
        auto row_sum_plain = [&](F2 part, float *rh) -> float {
            float v = __fadd_rn(f2_lo(part), f2_hi(part));
            const int width = SUB ? tpr : 32;
            for (int o = width >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if constexpr (!SUB) {
                const int nwarp = tpr >> 5;
                const int warp = threadIdx.x >> 5;
                if ((threadIdx.x & 31) == 0) rh[warp] = v;
                __syncthreads();
                int w = 1;
                while (w < nwarp) w <<= 1;
                const int i = threadIdx.x & (w - 1);
                v = i < nwarp ? rh[grp * nwarp + i] : 0.f;
                for (int o = w >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            }
            return v;
        };
        float mean = 0.f;
        if constexpr (LN) {
            mean = __fdiv_rn(row_sum_plain(ss2, red2_h), (float)p.H);
            // Squared deviations of this thread's elements (none past the row).
            const F2 nm2 = f2(-mean);
            ss2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const bool ok = live && k * tpr + lane < nvec;
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    const F2 d = f2_add(f2_bf16(h[k].w[i]), nm2);
                    if (ok) ss2 = f2_fma(d, d, ss2);
                }
            }
            if (p.mean != nullptr && live && lane == 0)
                p.mean[t] = mean;
        }
        float ssum;
        if constexpr (LN) ssum = row_sum_plain(ss2, red_h);
        else ssum = row_sum(ss2, red_h, red_l);
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ssum, (float)p.H), p.eps)));
        if (p.rstd != nullptr && live && lane == 0)
            p.rstd[t] = rstd;

        // ---------------- phase 4: epilogue -----------------------------------
        float scale_v = 1.f;
        if constexpr (OUT == OUT_Q || OUT == OUT_ADA_Q)
            scale_v = __ldg(p.scale);
        if constexpr (OUT == OUT_SILU_Q)
            scale_v = p.scale != nullptr ? __ldg(p.scale) : 1.f;
        const DivScale dsc(scale_v);            // IEEE division by the scale
        const F2 nmean2 = f2(-mean);
        const F2 rstd2 = f2(rstd);
        const F2 bias2 = f2(p.bias);

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            const bool ok = live && v < nvec;
            const int64_t c = (int64_t)v * VEC;
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
                const F2 w2 = W32 ? f2(wf[k][2 * i], wf[k][2 * i + 1]) : f2_bf16(wb[k].w[i]);
                if constexpr (LN)
                    o[i] = f2_fma(f2_mul(f2_add(f2_bf16(h[k].w[i]), nmean2), rstd2), w2,
                                  f2(bt[k][2 * i], bt[k][2 * i + 1]));
                else
                    o[i] = f2_mul(f2_mul(f2_bf16(h[k].w[i]), rstd2), f2_add(w2, bias2));
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
                    float a, b;
                    dsc.div(o[i], a, b);
                    cq[i] = pack_fp8<FP8K>(a, b);
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
                        p.bscale[(int64_t)(v >> 4) * p.ldT + t] = s;
                }
            } else if constexpr (OUT == OUT_SILU) {
                BVec<VEC> yv;
#pragma unroll
                for (int i = 0; i < NW; ++i) yv.w[i] = pack_bf16(silu_f32(f2_lo(o[i])), silu_f32(f2_hi(o[i])));
                if (ok) st_stream<VEC>(p.y + t * p.ldy + c, yv);
            } else if constexpr (OUT == OUT_SILU_Q) {
                uint32_t cq[NW];
                if (p.scale == nullptr) {      // the plain cast (no division by 1)
#pragma unroll
                    for (int i = 0; i < NW; ++i)
                        cq[i] = pack_fp8<0>(silu_f32(f2_lo(o[i])), silu_f32(f2_hi(o[i])));
                } else {
#pragma unroll
                    for (int i = 0; i < NW; ++i)
                        cq[i] = pack_fp8<0>(__fdiv_rn(silu_f32(f2_lo(o[i])), scale_v),
                                            __fdiv_rn(silu_f32(f2_hi(o[i])), scale_v));
                }
                if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
            } else {  // ADA: o * (1 + scale) + shift, one FP32 rounding (fma)
                const F2 one2 = f2(1.f);
                F2 ov[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i)
                    ov[i] = f2_fma(o[i], f2_add(one2, f2_bf16(sc[k].w[i])), f2_bf16(sh[k].w[i]));
                if constexpr (OUT == OUT_ADA) {
                    BVec<VEC> out;
#pragma unroll
                    for (int i = 0; i < NW; ++i) out.w[i] = bf16_f2(ov[i]);
                    if (ok) st_stream<VEC>(p.y + t * p.ldy + c, out);
                } else {
                    uint32_t cq[NW];
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        float a, b;
                        dsc.div(ov[i], a, b);
                        cq[i] = pack_fp8<0>(a, b);
                    }
                    if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
                }
                if (ok) st_stream<VEC>(p.gate_out + t * p.ldgo + c, gt[k]);
            }
        }
    };

    if constexpr (!LOOP) {
        const int64_t t = (int64_t)blockIdx.x * p.rpc + grp;
        load_row(t, xa, true);
        process(t);
    } else {
        static_assert(IN == IN_PLAIN, "the persistent form streams one input");
        load_weights();
        const int64_t stride = (int64_t)gridDim.x * p.rpc;
        const int64_t b0 = (int64_t)blockIdx.x * p.rpc;
        load_row(b0 + grp, xa, false);
        for (int64_t base = b0; base < p.T; base += stride) {
            BVec<VEC> xn[VPT];
            const bool more = base + stride < p.T;   // the same for the whole CTA
            if (more) load_row(base + stride + grp, xn, false);
            process(base + grp);
            if (more) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) xa[k] = xn[k];
            }
        }
    }
}

// Host-side launch of one instantiation.  The single-input variants run the
// persistent form on at most (resident CTAs per SM) x (SMs) CTAs; the
// residency of a block size is computed once and remembered.
template <int IN, bool W32, int OUT, int FP8K, int VEC, int VPT, bool SUB>
cudaError_t launch_fwd_inst(const FwdParams &p, cudaStream_t s)
{
    // Measured: the persistent form pays off for the plain row with the y and
    // static FP8 epilogues; SiLU (bound by its arithmetic) and LayerNorm
    // (gamma and beta) run faster in the one-row form.
    constexpr bool LOOP = IN == IN_PLAIN && (OUT == OUT_Y || OUT == OUT_Q);
    auto kern = k_rmsnorm_fwd<IN, W32, OUT, FP8K, VEC, VPT, SUB, LOOP>;
    const int threads = p.tpr * p.rpc;
    int64_t blocks = (p.T + p.rpc - 1) / p.rpc;
    if constexpr (LOOP) {
        static std::atomic<long long> cached{0};   // threads << 32 | CTAs per SM
        long long c = cached.load(std::memory_order_relaxed);
        int per_sm = (int)(c & 0xffffffff);
        if ((c >> 32) != threads || per_sm <= 0) {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) per_sm = 1;
            cached.store(((long long)threads << 32) | per_sm, std::memory_order_relaxed);
        }
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t cap = (int64_t)per_sm * sms;
        if (blocks > cap) blocks = cap;
    }
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(threads), 0, s, p);
}

// Dispatch over the row layouts the host chooser can return: SUB groups with
// VPT 1|2; multi-warp groups with VPT 2|4 (16-byte vectors) or 2|4|8|16
// (4-byte vectors), i.e. at most 32 elements per thread.
template <int IN, bool W32, int OUT, int FP8K, int VEC>
cudaError_t launch_fwd_vec(const FwdParams &p, int vpt, bool sub, cudaStream_t s)
{
    if (sub) {
        if (vpt == 1) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 1, true>(p, s);
        if (vpt == 2) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 2, true>(p, s);
    } else {
        if (vpt == 2) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 2, false>(p, s);
        if (vpt == 4) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 4, false>(p, s);
        if constexpr (VEC == 2) {
            if (vpt == 8) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 8, false>(p, s);
            if (vpt == 16) return launch_fwd_inst<IN, W32, OUT, FP8K, VEC, 16, false>(p, s);
        }
    }
    return cudaErrorInvalidConfiguration;
}

template <int IN, bool W32, int OUT, int FP8K>
cudaError_t launch_fwd(const FwdParams &p, int vec, int vpt, bool sub, cudaStream_t s)
{
    if (vec == 8) return launch_fwd_vec<IN, W32, OUT, FP8K, 8>(p, vpt, sub, s);
    if constexpr (OUT != OUT_BLOCK)
        if (vec == 2) return launch_fwd_vec<IN, W32, OUT, FP8K, 2>(p, vpt, sub, s);
    return cudaErrorInvalidConfiguration;
}

}  // namespace crmsn
