// fwd_block_ada.cu -- instantiations of the forward kernel with the 1x128
// block-quant epilogue and the AdaRMSNorm style epilogues.
#include "fwd.cuh"

namespace crmsn {

cudaError_t launch_fwd_block(const FwdParams &p, const Layout &L, cudaStream_t s)
{
    return launch_fwd<IN_RESIDUAL, WK_MIX, OUT_BLOCK, 0>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_ada(const FwdParams &p, bool gated_fp8, const Layout &L, cudaStream_t s)
{
    if (gated_fp8) return launch_fwd<IN_GATED, WK_MIX, OUT_ADA_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN_PLAIN, WK_MIX, OUT_ADA, 0>(p, L.vec, L.vpt, L.sub, s);
}

}  // namespace crmsn
