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
#pragma once

#include "launch.h"

namespace crmsn {

template <int IN, bool W32, int OUT, int FP8K, int VEC, int VPT, bool SUB>
__global__ void __launch_bounds__(kFwdMaxThreads)
k_rmsnorm_fwd(const FwdParams p)
{
    constexpr int NW = VEC / 2;
    constexpr bool ADA = (OUT == OUT_ADA || OUT == OUT_ADA_Q);
    __shared__ float red_h[32], red_l[32];

    const int tpr = p.tpr;
    const int grp = threadIdx.x / tpr;
    const int lane = threadIdx.x - grp * tpr;
    const int64_t t = (int64_t)blockIdx.x * p.rpc + grp;
    const bool live = t < p.T;
    const int nvec = p.H / VEC;

    // ---------------- phase 1: issue every load of the row ----------------
    BVec<VEC> xa[VPT], ra[VPT], ga[VPT];
    BVec<VEC> sc[VPT], sh[VPT], gt[VPT];
    BVec<VEC> wb[VPT];
    float wf[VPT][VEC];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * tpr + lane;
        if (live && v < nvec) {
            const int64_t c = (int64_t)v * VEC;
            xa[k] = ld_stream<VEC>(p.x + t * p.ldx + c);
            if constexpr (IN != IN_PLAIN)
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
            if constexpr (W32)
                ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, wf[k]);
            else
                wb[k] = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                xa[k].w[i] = 0u; ra[k].w[i] = 0u; ga[k].w[i] = 0u;
                sc[k].w[i] = 0u; sh[k].w[i] = 0u; gt[k].w[i] = 0u; wb[k].w[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < VEC; ++i) wf[k][i] = 0.f;
        }
    }

    // ---------------- phase 2: normalised input h, sum of squares ---------
    BVec<VEC> h[VPT];
    F2 ss2 = f2(0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t xw = xa[k].w[i];
            uint32_t hw;
            if constexpr (IN == IN_PLAIN) {
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
            // h^2 is exact in FP32, so the fma rounds only the accumulation.
            const F2 h2 = f2_bf16(hw);
            ss2 = f2_fma(h2, h2, ss2);
        }
        if constexpr (IN != IN_PLAIN) {
            const int v = k * tpr + lane;
            if (live && v < nvec)
                st_stream<VEC>(p.hn + t * p.ldh + (int64_t)v * VEC, h[k]);
        }
    }

    // ---------------- phase 3: row reduction -> rstd ----------------------
    float sh_, sl_;
    two_sum(f2_lo(ss2), f2_hi(ss2), sh_, sl_);
    if constexpr (SUB) {
        pair_reduce_lanes(sh_, sl_, tpr);
    } else {
        // Butterfly within each warp, then across the group's warps: short
        // latency for these short-lived CTAs.
        pair_reduce_lanes(sh_, sl_, 32);
        const int nwarp = tpr >> 5;
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            red_h[warp] = sh_;
            red_l[warp] = sl_;
        }
        __syncthreads();
        pair_reduce_warps(sh_, sl_, red_h, red_l, grp * nwarp, nwarp);
    }
    const float ssum = __fadd_rn(sh_, sl_);
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ssum, (float)p.H), p.eps)));
    if (p.rstd != nullptr && live && lane == 0)
        p.rstd[t] = rstd;

    // ---------------- phase 4: epilogue -----------------------------------
    float scale_v = 1.f;
    if constexpr (OUT == OUT_Q || OUT == OUT_ADA_Q)
        scale_v = __ldg(p.scale);
    const F2 rstd2 = f2(rstd);
    const F2 bias2 = f2(p.bias);

#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * tpr + lane;
        const bool ok = live && v < nvec;
        const int64_t c = (int64_t)v * VEC;
        F2 o[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const F2 w2 = W32 ? f2(wf[k][2 * i], wf[k][2 * i + 1]) : f2_bf16(wb[k].w[i]);
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
            for (int i = 0; i < NW; ++i)
                cq[i] = pack_fp8<FP8K>(__fdiv_rn(f2_lo(o[i]), scale_v), __fdiv_rn(f2_hi(o[i]), scale_v));
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
            uint32_t cq[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                if (s > 0.f)
                    cq[i] = pack_fp8<0>(__fdiv_rn(bf_lo(nv.w[i]), s), __fdiv_rn(bf_hi(nv.w[i]), s));
                else
                    cq[i] = 0u;
            }
            if (ok) {
                st_fp8<VEC>(p.q + t * p.ldq + c, cq);
                if ((v & 15) == 0)
                    p.bscale[(int64_t)(v >> 4) * p.ldT + t] = s;
            }
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
                for (int i = 0; i < NW; ++i)
                    cq[i] = pack_fp8<0>(__fdiv_rn(f2_lo(ov[i]), scale_v), __fdiv_rn(f2_hi(ov[i]), scale_v));
                if (ok) st_fp8<VEC>(p.q + t * p.ldq + c, cq);
            }
            if (ok) st_stream<VEC>(p.gate_out + t * p.ldgo + c, gt[k]);
        }
    }
}

// Host-side launch of one instantiation.
template <int IN, bool W32, int OUT, int FP8K, int VEC, int VPT, bool SUB>
cudaError_t launch_fwd_inst(const FwdParams &p, cudaStream_t s)
{
    const int threads = p.tpr * p.rpc;
    const int64_t blocks = (p.T + p.rpc - 1) / p.rpc;
    k_rmsnorm_fwd<IN, W32, OUT, FP8K, VEC, VPT, SUB><<<(unsigned)blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
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
