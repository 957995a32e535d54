// bwd.cu -- RMSNorm backward: dx per row and a deterministic FP32 dw.
//
// Source: "FlashInfer normalization operator guide" 6.1-6.3 and the
// "cake_rmsnorm_det_train_forward" Notes:
//   m    = mean(g * w * x)
//   dx   = bf16(rstd*g*w - x*rstd^3*m (+ g_residual))
//   dw   = sum_t g * x * rstd, bitwise reproducible for a given T and SM count.
//
// Design (GB300): CTA c owns the contiguous row chunk [c*T/n, (c+1)*T/n) of a
// fixed chunk table (n = chunks, a function of T and the SM count).  Each
// thread owns the same columns in every row, so it keeps the effective weight
// and a compensated (TwoSum) dw accumulator per column in registers while it
// walks its chunk; the next row's g, x and rstd are loaded before the current
// row is reduced, so one row is always in flight behind the arithmetic.  At
// the end the CTA writes one FP32 partial row; a second, small kernel adds the
// partial rows of every column in chunk order (again compensated).  The
// second kernel is launched with programmatic dependent launch and waits on
// the first grid with griddepcontrol.wait, a hardware dependency rather than
// a spin loop.
#include "launch.h"

namespace crmsn {

template <bool W32, bool GRES, int VEC, int VPT, bool SUB>
__global__ void __launch_bounds__(kBwdMaxThreads, 1)
k_rmsnorm_bwd(const BwdParams p)
{
    constexpr int NW = VEC / 2;
    __shared__ float red_h[32], red_l[32];
    extern __shared__ float dyn_smem[];   // w_eff [H], then [rpc-1][H][2] when rpc > 1
    float *comb = dyn_smem;

    const int tpr = p.tpr;
    const int rpc = p.rpc;
    const int grp = threadIdx.x / tpr;
    const int lane = threadIdx.x - grp * tpr;
    const int nvec = p.H / VEC;
    const int64_t r0 = (int64_t)blockIdx.x * p.T / p.nchunk;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * p.T / p.nchunk;
    const int64_t iters = (r1 - r0 + rpc - 1) / rpc;

    // Effective weight f32(w + bias) of this thread's columns, fixed for the
    // whole chunk, kept in shared memory (each thread reads back only the
    // columns it wrote, so no barrier is needed) to leave the registers to
    // the row data and the dw accumulators.
    float *wsm = comb;
    comb += p.H;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * tpr + lane;
        if (grp == 0 && v < nvec) {
            const int64_t c = (int64_t)v * VEC;
            if constexpr (W32) {
                float f[VEC];
                ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, f);
#pragma unroll
                for (int i = 0; i < VEC; ++i) wsm[c + i] = __fadd_rn(f[i], p.bias);
            } else {
                BVec<VEC> wb = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    wsm[c + 2 * i] = __fadd_rn(bf_lo(wb.w[i]), p.bias);
                    wsm[c + 2 * i + 1] = __fadd_rn(bf_hi(wb.w[i]), p.bias);
                }
            }
        }
    }
    if (rpc > 1) __syncthreads();   // other row groups read group 0's copy
    auto weff = [&](int k, int e) -> float {
        const int v = k * tpr + lane;
        return v < nvec ? wsm[v * VEC + e] : 0.f;
    };

    float acc[VPT][VEC], cmp[VPT][VEC];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int i = 0; i < VEC; ++i) { acc[k][i] = 0.f; cmp[k][i] = 0.f; }

    BVec<VEC> gc[VPT], xc[VPT], rc[VPT];
    float rsc = 0.f;
    auto load_row = [&](int64_t t, bool live, BVec<VEC> (&gv)[VPT], BVec<VEC> (&xv)[VPT],
                        BVec<VEC> (&rv)[VPT], float &rs) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            if (live && v < nvec) {
                const int64_t c = (int64_t)v * VEC;
                gv[k] = ld_stream<VEC>(p.g + t * p.ldg + c);
                xv[k] = ld_stream<VEC>(p.x + t * p.ldx + c);
                if constexpr (GRES) rv[k] = ld_stream<VEC>(p.gres + t * p.ldgr + c);
            } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) { gv[k].w[i] = 0u; xv[k].w[i] = 0u; rv[k].w[i] = 0u; }
            }
        }
        rs = live ? __ldg(p.rstd + t) : 0.f;
    };

    // Rows of up to 16 elements per thread prefetch the next row into a second
    // register set; wider rows already keep a whole row per CTA in flight.
    constexpr bool PF = VPT * VEC <= 16;
    if constexpr (PF) load_row(r0 + grp, (r0 + grp) < r1, gc, xc, rc, rsc);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t t = r0 + grp + it * rpc;
        const bool live = t < r1;
        BVec<VEC> gn[VPT], xn[VPT], rn[VPT];
        float rsn = 0.f;
        const int64_t tn = t + rpc;
        if constexpr (PF)
            load_row(tn, (it + 1 < iters) && tn < r1, gn, xn, rn, rsn);
        else
            load_row(t, live, gc, xc, rc, rsc);

        // m = mean(g * w * x): FP32 per thread, compensated across threads.
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                dot = __fmaf_rn(__fmul_rn(bf_lo(gc[k].w[i]), weff(k, 2 * i)), bf_lo(xc[k].w[i]), dot);
                dot = __fmaf_rn(__fmul_rn(bf_hi(gc[k].w[i]), weff(k, 2 * i + 1)), bf_hi(xc[k].w[i]), dot);
            }
        float dh = dot, dl = 0.f;
        if constexpr (SUB) {
            pair_reduce_lanes(dh, dl, tpr);
        } else {
            pair_reduce_lanes(dh, dl, 32);
            const int nwarp = tpr >> 5;
            const int warp = threadIdx.x >> 5;
            if ((threadIdx.x & 31) == 0) { red_h[warp] = dh; red_l[warp] = dl; }
            __syncthreads();
            const int w0 = grp * nwarp;
            dh = red_h[w0];
            dl = red_l[w0];
            for (int i = 1; i < nwarp; ++i) pair_add(dh, dl, red_h[w0 + i], red_l[w0 + i]);
            __syncthreads();   // red_* is rewritten by the next row
        }
        const float m = __fdiv_rn(__fadd_rn(dh, dl), (float)p.H);
        const float rs = rsc;
        const float c3 = __fmul_rn(__fmul_rn(__fmul_rn(rs, rs), rs), m);

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            float d[VEC];
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                const float g0 = bf_lo(gc[k].w[i]), g1 = bf_hi(gc[k].w[i]);
                const float x0 = bf_lo(xc[k].w[i]), x1 = bf_hi(xc[k].w[i]);
                d[2 * i] = __fmaf_rn(-x0, c3, __fmul_rn(rs, __fmul_rn(g0, weff(k, 2 * i))));
                d[2 * i + 1] = __fmaf_rn(-x1, c3, __fmul_rn(rs, __fmul_rn(g1, weff(k, 2 * i + 1))));
                if constexpr (GRES) {
                    d[2 * i] = __fadd_rn(d[2 * i], bf_lo(rc[k].w[i]));
                    d[2 * i + 1] = __fadd_rn(d[2 * i + 1], bf_hi(rc[k].w[i]));
                }
                // dw term g*x*rstd: g*x is exact in FP32; TwoSum keeps the
                // accumulation error in cmp.
                const float e0 = __fmul_rn(__fmul_rn(g0, x0), rs);
                const float e1 = __fmul_rn(__fmul_rn(g1, x1), rs);
                float s, err;
                two_sum(acc[k][2 * i], e0, s, err);
                acc[k][2 * i] = s;
                cmp[k][2 * i] = __fadd_rn(cmp[k][2 * i], err);
                two_sum(acc[k][2 * i + 1], e1, s, err);
                acc[k][2 * i + 1] = s;
                cmp[k][2 * i + 1] = __fadd_rn(cmp[k][2 * i + 1], err);
            }
            if (live && v < nvec) {
                BVec<VEC> o;
#pragma unroll
                for (int i = 0; i < NW; ++i) o.w[i] = pack_bf16(d[2 * i], d[2 * i + 1]);
                st_stream<VEC>(p.dx + t * p.lddx + (int64_t)v * VEC, o);
            }
        }
        if constexpr (PF) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) { gc[k] = gn[k]; xc[k] = xn[k]; rc[k] = rn[k]; }
            rsc = rsn;
        }
    }

    // Combine the CTA's row groups in group order, then write the partial row.
    if (rpc > 1) {
        if (grp > 0) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * tpr + lane;
                if (v < nvec)
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        float *slot = comb + ((int64_t)(grp - 1) * p.H + (int64_t)v * VEC + i) * 2;
                        slot[0] = acc[k][i];
                        slot[1] = cmp[k][i];
                    }
            }
        }
        __syncthreads();
        if (grp == 0) {
            for (int gi = 1; gi < rpc; ++gi)
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * tpr + lane;
                    if (v < nvec)
#pragma unroll
                        for (int i = 0; i < VEC; ++i) {
                            const float *slot = comb + ((int64_t)(gi - 1) * p.H + (int64_t)v * VEC + i) * 2;
                            pair_add(acc[k][i], cmp[k][i], slot[0], slot[1]);
                        }
                }
        }
    }
    if (grp == 0) {
        float *prow = p.part + (int64_t)blockIdx.x * p.H;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            if (v < nvec)
#pragma unroll
                for (int i = 0; i < VEC; ++i)
                    prow[(int64_t)v * VEC + i] = __fadd_rn(acc[k][i], cmp[k][i]);
        }
    }
    // Let the dependent reduce grid get scheduled; it still waits for this
    // whole grid (and its memory) with griddepcontrol.wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// dw[j] = sum over chunks c (in order) of part[c][j], compensated.  A block
// covers 32*CPT columns; its NS warps each sum a fixed contiguous range of
// chunks, and warp 0 adds the NS pair sums in warp order.
template <int CPT>
__global__ void __launch_bounds__(512)
k_dw_reduce(const float *__restrict__ part, int nchunk, int H, float *__restrict__ dw)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float sh_h[16][32 * CPT], sh_l[16][32 * CPT];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int ns = blockDim.x >> 5;
    const int col = (blockIdx.x * 32 + lane) * CPT;
    const int c0 = (int)((int64_t)warp * nchunk / ns);
    const int c1 = (int)((int64_t)(warp + 1) * nchunk / ns);
    float h[CPT], l[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) { h[i] = 0.f; l[i] = 0.f; }
    if (col < H) {
#pragma unroll 4
        for (int c = c0; c < c1; ++c) {
            const float *src = part + (int64_t)c * H + col;
            float v[CPT];
            if constexpr (CPT == 4) {
                float4 f = __ldcg(reinterpret_cast<const float4 *>(src));
                v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
            } else {
                float2 f = __ldcg(reinterpret_cast<const float2 *>(src));
                v[0] = f.x; v[1] = f.y;
            }
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                float s, e;
                two_sum(h[i], v[i], s, e);
                h[i] = s;
                l[i] = __fadd_rn(l[i], e);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        sh_h[warp][lane * CPT + i] = h[i];
        sh_l[warp][lane * CPT + i] = l[i];
    }
    __syncthreads();
    if (warp == 0 && col < H) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            float a = sh_h[0][lane * CPT + i], b = sh_l[0][lane * CPT + i];
            for (int w = 1; w < ns; ++w) pair_add(a, b, sh_h[w][lane * CPT + i], sh_l[w][lane * CPT + i]);
            dw[col + i] = __fadd_rn(a, b);
        }
    }
}

static cudaError_t launch_dw_reduce(const float *part, int nchunk, int H, float *dw, cudaStream_t s)
{
    const int cpt = (H % 4 == 0) ? 4 : 2;
    const int ns = nchunk >= 128 ? 16 : (nchunk >= 16 ? 8 : 1);
    const unsigned blocks = (unsigned)((H + 32 * cpt - 1) / (32 * cpt));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(32 * ns);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = (cpt == 4) ? cudaLaunchKernelEx(&cfg, k_dw_reduce<4>, part, nchunk, H, dw)
                               : cudaLaunchKernelEx(&cfg, k_dw_reduce<2>, part, nchunk, H, dw);
    if (e != cudaSuccess) {
        // Without the attribute the launch is an ordinary stream-ordered one;
        // griddepcontrol.wait then returns at once.
        (void)cudaGetLastError();
        cfg.numAttrs = 0;
        e = (cpt == 4) ? cudaLaunchKernelEx(&cfg, k_dw_reduce<4>, part, nchunk, H, dw)
                       : cudaLaunchKernelEx(&cfg, k_dw_reduce<2>, part, nchunk, H, dw);
    }
    return e;
}

template <bool W32, bool GRES, int VEC, int VPT, bool SUB>
static cudaError_t launch_bwd_inst(BwdParams p, int sms, float *dw, cudaStream_t s)
{
    const int threads = p.tpr * p.rpc;
    const size_t smem = ((size_t)p.H + (size_t)(p.rpc - 1) * p.H * 2) * sizeof(float);
    auto kern = k_rmsnorm_bwd<W32, GRES, VEC, VPT, SUB>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > kBwdMaxCtasPerSm) per_sm = kBwdMaxCtasPerSm;
    const int64_t by_rows = (p.T + p.rpc - 1) / p.rpc;
    const int64_t cap = (int64_t)per_sm * sms;
    p.nchunk = (int)(by_rows < cap ? by_rows : cap);
    kern<<<p.nchunk, threads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dw_reduce(p.part, p.nchunk, p.H, dw, s);
}

// Layouts: SUB groups with VPT 1|2; multi-warp groups with VPT 1|2|4 (16-byte
// vectors) or 1|2|4|8|16 (4-byte vectors).
template <bool W32, bool GRES, int VEC>
static cudaError_t launch_bwd_vec(const BwdParams &p, const Layout &L, int sms, float *dw,
                                  cudaStream_t s)
{
    if (L.sub) {
        if (L.vpt == 1) return launch_bwd_inst<W32, GRES, VEC, 1, true>(p, sms, dw, s);
        if (L.vpt == 2) return launch_bwd_inst<W32, GRES, VEC, 2, true>(p, sms, dw, s);
    } else {
        if (L.vpt == 1) return launch_bwd_inst<W32, GRES, VEC, 1, false>(p, sms, dw, s);
        if (L.vpt == 2) return launch_bwd_inst<W32, GRES, VEC, 2, false>(p, sms, dw, s);
        if (L.vpt == 4) return launch_bwd_inst<W32, GRES, VEC, 4, false>(p, sms, dw, s);
        if constexpr (VEC == 2) {
            if (L.vpt == 8) return launch_bwd_inst<W32, GRES, VEC, 8, false>(p, sms, dw, s);
            if (L.vpt == 16) return launch_bwd_inst<W32, GRES, VEC, 16, false>(p, sms, dw, s);
        }
    }
    return cudaErrorInvalidConfiguration;
}

template <bool W32, bool GRES>
static cudaError_t launch_bwd_w(const BwdParams &p, const Layout &L, int sms, float *dw,
                                cudaStream_t s)
{
    if (L.vec == 8) return launch_bwd_vec<W32, GRES, 8>(p, L, sms, dw, s);
    if (L.vec == 2) return launch_bwd_vec<W32, GRES, 2>(p, L, sms, dw, s);
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_bwd(BwdParams p, bool w32, bool gres, const Layout &L, int sms, float *dw,
                       cudaStream_t s)
{
    if (w32) return gres ? launch_bwd_w<true, true>(p, L, sms, dw, s)
                         : launch_bwd_w<true, false>(p, L, sms, dw, s);
    return gres ? launch_bwd_w<false, true>(p, L, sms, dw, s)
                : launch_bwd_w<false, false>(p, L, sms, dw, s);
}

}  // namespace crmsn
