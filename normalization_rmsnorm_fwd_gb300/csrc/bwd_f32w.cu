// bwd_f32w.cu -- backward instantiations for an FP32 weight.
#include "bwd.cuh"

namespace crmsn {

cudaError_t launch_bwd_f32w(const BwdParams &p, bool gres, const Layout &L, int sms, int *nchunk,
                            cudaStream_t s)
{
    return launch_bwd_weight<true>(p, gres, L, sms, nchunk, s);
}

}  // namespace crmsn
