// bwd_reduce.cu -- the fixed-order reduction of the backward's per-chunk dw
// partial rows, and the backward launch sequence (partials kernel, then this
// reduction with programmatic dependent launch).
#include "launch.h"

namespace crmsn {

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

cudaError_t launch_bwd(BwdParams p, bool w32, bool gres, const Layout &L, int sms, float *dw,
                       cudaStream_t s)
{
    int nchunk = 0;
    cudaError_t e = w32 ? launch_bwd_f32w(p, gres, L, sms, &nchunk, s)
                        : launch_bwd_bf16w(p, gres, L, sms, &nchunk, s);
    if (e != cudaSuccess) return e;
    return launch_dw_reduce(p.part, nchunk, p.H, dw, s);
}

}  // namespace crmsn
