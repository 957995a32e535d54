// fwd_silu_ln.cu -- instantiations of the forward kernel for RMSNorm + SiLU
// (fused_rmsnorm_silu: BF16 or E4M3 output) and for LayerNorm (layernorm:
// BF16 output; layernorm_quant: E4M3FN or E5M2 output).
#include "fwd.cuh"

namespace crmsn {

template <int OUT>
static cudaError_t go(const FwdParams &p, int wk, const Layout &L, cudaStream_t s)
{
    if (wk == WK_MIX) return launch_fwd<IN_PLAIN, WK_MIX, OUT, 0>(p, L.vec, L.vpt, L.sub, s);
    if (wk == WK_BF16) return launch_fwd<IN_PLAIN, WK_BF16, OUT, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN_PLAIN, WK_F32, OUT, 0>(p, L.vec, L.vpt, L.sub, s);
}

cudaError_t launch_fwd_silu(const FwdParams &p, int wk, bool fp8, const Layout &L, cudaStream_t s)
{
    return fp8 ? go<OUT_SILU_Q>(p, wk, L, s) : go<OUT_SILU>(p, wk, L, s);
}

// gamma and beta are FP32 (the weight kind is not used by LayerNorm rows).
cudaError_t launch_fwd_layernorm(const FwdParams &p, int fp8k, const Layout &L, cudaStream_t s)
{
    if (fp8k < 0) return launch_fwd<IN_LAYERNORM, WK_F32, OUT_Y, 0>(p, L.vec, L.vpt, L.sub, s);
    if (fp8k == 0) return launch_fwd<IN_LAYERNORM, WK_F32, OUT_Q, 0>(p, L.vec, L.vpt, L.sub, s);
    return launch_fwd<IN_LAYERNORM, WK_F32, OUT_Q, 1>(p, L.vec, L.vpt, L.sub, s);
}

}  // namespace crmsn
