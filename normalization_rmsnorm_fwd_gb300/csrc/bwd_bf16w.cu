// bwd_bf16w.cu -- backward instantiations for a BF16 weight, without g_residual.
#include "bwd.cuh"

namespace crmsn {

cudaError_t launch_bwd_bf16w_plain(const BwdParams &p, const Layout &L, int sms, int *nchunk,
                                   cudaStream_t s)
{
    return launch_bwd_weight<false, false>(p, L, sms, nchunk, s);
}

}  // namespace crmsn
