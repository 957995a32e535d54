// fwd_silu_ln.cu -- instantiations of the forward kernel for RMSNorm + SiLU
// (fused_rmsnorm_silu: BF16 or E4M3 output) and for LayerNorm (layernorm:
// BF16 output; layernorm_quant: E4M3FN or E5M2 output).
#include "fwd.cuh"

namespace crmsn {

cudaError_t launch_fwd_silu(const FwdParams &p, bool w32, bool fp8, const Layout &L, cudaStream_t s)
{
    if (fp8)
        return w32 ? launch_fwd<IN_PLAIN, true, OUT_SILU_Q, 0>(p, L.vec, L.vpt, L.sub, s)
                   : launch_fwd<IN_PLAIN, false, OUT_SILU_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return w32 ? launch_fwd<IN_PLAIN, true, OUT_SILU, 0>(p, L.vec, L.vpt, L.sub, s)
               : launch_fwd<IN_PLAIN, false, OUT_SILU, 0>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_layernorm(const FwdParams &p, int fp8k, const Layout &L, cudaStream_t s)
{
    if (fp8k < 0) return launch_fwd<IN_LAYERNORM, true, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
    if (fp8k == 0) return launch_fwd<IN_LAYERNORM, true, OUT_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN_LAYERNORM, true, OUT_Q, 1>(p, L.vec, L.vpt, L.sub, s);
}

}  // namespace crmsn
