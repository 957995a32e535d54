// bwd_bf16w_gres.cu -- backward instantiations for a BF16 weight, with g_residual.
#include "bwd.cuh"

namespace crmsn {

cudaError_t launch_bwd_bf16w_gres(const BwdParams &p, const Layout &L, int sms, int *nchunk,
                                  cudaStream_t s)
{
    return launch_bwd_weight<false, true>(p, L, sms, nchunk, s);
}

}  // namespace crmsn
