// fwd_q.cu -- instantiations of the forward kernel with the static-scale FP8
// epilogue (rmsnorm_quant, fused_add_rmsnorm_quant; E4M3FN and E5M2).
#include "fwd.cuh"

namespace crmsn {

template <int IN, int WK>
static cudaError_t go(const FwdParams &p, int fp8k, const Layout &L, cudaStream_t s)
{
    if (fp8k == 0) return launch_fwd<IN, WK, OUT_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN, WK, OUT_Q, 1>(p, L.vec, L.vpt, L.sub, s);
}

template <int IN>
static cudaError_t go_w(const FwdParams &p, int wk, int fp8k, const Layout &L, cudaStream_t s)
{
    if (wk == WK_MIX) return go<IN, WK_MIX>(p, fp8k, L, s);
    if (wk == WK_BF16) return go<IN, WK_BF16>(p, fp8k, L, s);
    return go<IN, WK_F32>(p, fp8k, L, s);
}

cudaError_t launch_fwd_q(const FwdParams &p, int in, int wk, int fp8k, const Layout &L,
                         cudaStream_t s)
{
    if (in == IN_PLAIN) return go_w<IN_PLAIN>(p, wk, fp8k, L, s);
    if (in == IN_RESIDUAL) return go_w<IN_RESIDUAL>(p, wk, fp8k, L, s);
    return cudaErrorInvalidValue;
}

}  // namespace crmsn
