// fwd_y.cu -- instantiations of the forward kernel with the BF16 y epilogue
// (rmsnorm, gemma_rmsnorm, fused_add_rmsnorm, zero-centred FP32 weight).
#include "fwd.cuh"

namespace crmsn {

template <int IN>
static cudaError_t go(const FwdParams &p, int wk, const Layout &L, cudaStream_t s)
{
    if (wk == WK_MIX) return launch_fwd<IN, WK_MIX, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
    if (wk == WK_BF16) return launch_fwd<IN, WK_BF16, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN, WK_F32, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_y(const FwdParams &p, int in, int wk, const Layout &L, cudaStream_t s)
{
    if (in == IN_PLAIN) return go<IN_PLAIN>(p, wk, L, s);
    if (in == IN_RESIDUAL) return go<IN_RESIDUAL>(p, wk, L, s);
    return cudaErrorInvalidValue;
}

}  // namespace crmsn
