// fwd_y.cu -- instantiations of the forward kernel with the BF16 y epilogue
// (rmsnorm, gemma_rmsnorm, fused_add_rmsnorm, zero-centred FP32 weight).
#include "fwd.cuh"

namespace crmsn {

template <int IN, bool W32>
static cudaError_t go(const FwdParams &p, const Layout &L, cudaStream_t s)
{
    return launch_fwd<IN, W32, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_y(const FwdParams &p, int in, bool w32, const Layout &L, cudaStream_t s)
{
    if (in == IN_PLAIN) return w32 ? go<IN_PLAIN, true>(p, L, s) : go<IN_PLAIN, false>(p, L, s);
    if (in == IN_RESIDUAL) return w32 ? go<IN_RESIDUAL, true>(p, L, s) : go<IN_RESIDUAL, false>(p, L, s);
    return cudaErrorInvalidValue;
}

}  // namespace crmsn
