// bwd_bf16w.cu -- backward instantiations for a BF16 weight.
#include "bwd.cuh"

namespace crmsn {

cudaError_t launch_bwd_bf16w(const BwdParams &p, bool gres, const Layout &L, int sms, int *nchunk,
                             cudaStream_t s)
{
    return launch_bwd_weight<false>(p, gres, L, sms, nchunk, s);
}

}  // namespace crmsn
