// bwd_reduce.cu -- the fixed-order reduction of the backward's per-chunk dw
// partial rows, and the backward launch sequence (partials kernel, then this
// reduction; every launch uses programmatic dependent launch).  In the
// column form the backward kernel writes dw itself and this reduction is not
// launched.
#include "launch.h"

namespace crmsn {

// dw[j] = sum over chunks c of part[c][j], compensated, in a fixed order.
// A block covers 32 consecutive columns, one per lane, with kReduceWarps
// warps; warp w sums the contiguous chunk range [w*n/W, (w+1)*n/W) in chunk
// order, issuing all its loads (up to kBatch at a time) before adding them.
// The warps' pairs then meet in a fixed butterfly: warp j takes column j,
// lane i holding warp i's pair.  One round trip to L2 (where the partials
// were just written) for up to kBatch*kReduceWarps chunks, and no serial
// combine.
constexpr int kReduceWarps = 32;
constexpr int kBatch = 16;

#ifdef CRMSN_DEBUG
#define DW_REDUCE_DEBUG_PARAM , const DebugRanges dbg
#define DW_REDUCE_DEBUG_ARG , p.dbg
#else
#define DW_REDUCE_DEBUG_PARAM
#define DW_REDUCE_DEBUG_ARG
#endif

__global__ void __launch_bounds__(32 * kReduceWarps)
k_dw_reduce(const float *__restrict__ part, int nchunk, int H, float *__restrict__ dw DW_REDUCE_DEBUG_PARAM)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    CRMSN_DEBUG_ENTER(dbg);
    __shared__ float sh_h[kReduceWarps][33], sh_l[kReduceWarps][33];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    const int c0 = (int)((int64_t)warp * nchunk / kReduceWarps);
    const int c1 = (int)((int64_t)(warp + 1) * nchunk / kReduceWarps);
    float h = 0.f, l = 0.f;
    if (col < H) {
        for (int c = c0; c < c1; c += kBatch) {
            float v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                v[i] = (c + i < c1 && dbg_global(part + (int64_t)(c + i) * H + col, 4, false))
                           ? __ldcg(part + (int64_t)(c + i) * H + col) : 0.f;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                float s, e;
                two_sum(h, v[i], s, e);
                h = s;
                l = __fadd_rn(l, e);
            }
        }
    }
    sh_h[warp][lane] = h;
    sh_l[warp][lane] = l;
    __syncthreads();
    // Warp j: column j of the block; lane i: warp i's pair.
    float a = sh_h[lane][warp], b = sh_l[lane][warp];
    pair_reduce_lanes(a, b, 32);
    const int out = blockIdx.x * 32 + warp;
    if (lane == 0 && out < H) st_f32(dw + out, __fadd_rn(a, b));
}

static cudaError_t launch_dw_reduce(const BwdParams &p, int nchunk, float *dw, cudaStream_t s)
{
    return launch_pdl(k_dw_reduce, dim3((unsigned)((p.H + 31) / 32)), dim3(32 * kReduceWarps), 0, s,
                      (const float *)p.part, nchunk, p.H, dw DW_REDUCE_DEBUG_ARG);
}

cudaError_t launch_bwd(BwdParams p, bool w32, bool gres, const Layout &L, int sms, float *dw,
                       cudaStream_t s)
{
    int nchunk = 0;
    cudaError_t e = w32 ? (gres ? launch_bwd_f32w_gres(p, L, sms, &nchunk, s)
                                : launch_bwd_f32w_plain(p, L, sms, &nchunk, s))
                        : (gres ? launch_bwd_bf16w_gres(p, L, sms, &nchunk, s)
                                : launch_bwd_bf16w_plain(p, L, sms, &nchunk, s));
    if (e != cudaSuccess || p.ncols > 0) return e;
    return launch_dw_reduce(p, nchunk, dw, s);
}

}  // namespace crmsn
