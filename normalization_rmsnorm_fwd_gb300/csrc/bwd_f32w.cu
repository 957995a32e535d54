// bwd_f32w.cu -- backward instantiations for an FP32 weight, without g_residual.
#include "bwd.cuh"

namespace crmsn {

cudaError_t launch_bwd_f32w_plain(const BwdParams &p, const Layout &L, int sms, int *nchunk,
                                  cudaStream_t s)
{
    return launch_bwd_weight<true, false>(p, L, sms, nchunk, s);
}

}  // namespace crmsn
