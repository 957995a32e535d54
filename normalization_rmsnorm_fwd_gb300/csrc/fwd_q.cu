// fwd_q.cu -- instantiations of the forward kernel with the static-scale FP8
// epilogue (rmsnorm_quant, fused_add_rmsnorm_quant; E4M3FN and E5M2).
#include "fwd.cuh"

namespace crmsn {

template <int IN, bool W32>
static cudaError_t go(const FwdParams &p, int fp8k, const Layout &L, cudaStream_t s)
{
    if (fp8k == 0) return launch_fwd<IN, W32, OUT_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN, W32, OUT_Q, 1>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_q(const FwdParams &p, int in, bool w32, int fp8k, const Layout &L,
                         cudaStream_t s)
{
    if (in == IN_PLAIN)
        return w32 ? go<IN_PLAIN, true>(p, fp8k, L, s) : go<IN_PLAIN, false>(p, fp8k, L, s);
    if (in == IN_RESIDUAL)
        return w32 ? go<IN_RESIDUAL, true>(p, fp8k, L, s) : go<IN_RESIDUAL, false>(p, fp8k, L, s);
    return cudaErrorInvalidValue;
}

}  // namespace crmsn
