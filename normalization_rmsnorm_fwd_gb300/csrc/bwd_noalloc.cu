// bwd_noalloc.cu -- rmsnorm_bwd_noalloc: the backward with built-in scratch.
//
// Some callers cannot hand the library a workspace: an inference engine or
// plugin host that plans every device buffer ahead of time and forbids
// allocating inside an operation, or a plain C caller with no device
// allocator of its own, for whom a cudaMalloc per call would also stall the
// whole device.  This entry point runs the same backward as rmsnorm_bwd but
// takes its scratch (the per-chunk dw partial rows) from a fixed array that
// lives in the library's own device memory, so the call allocates nothing.
//
// The array is a file-scope __device__ variable of kScratchBytes; every GPU
// that loads the library keeps it until the process exits.  Host code never
// uses the array's name as a pointer (on the host it is only a stand-in):
// the first call on each device looks up its device address with
// cudaGetSymbolAddress while that device is current, and later calls reuse
// the cached address (valid in the device's primary context only: a
// cudaDeviceReset or a non-primary context would need a new lookup, which
// the header documents as unsupported).  All calls on a device share the one array, so calls
// that run at the same time on the GPU (different streams, or different host
// threads) overwrite each other's scratch and race; serialise them on one
// stream.  The scratch needs no initial value: the backward writes every
// partial it later reads.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "crmsnorm.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices];   // device address of g_bwd_scratch, per device

// Device address of the scratch array on the current device (looked up once).
crmsn_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return CRMSN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return CRMSN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CRMSN_OK;
}

}  // namespace

extern "C" crmsn_status rmsnorm_bwd_noalloc(const void *g, int64_t ldg, const void *x, int64_t ldx,
                                            const void *w, int w_dtype, float weight_bias,
                                            const float *rstd, const void *g_residual,
                                            int64_t ldgr, int64_t T, int64_t H, void *dx,
                                            int64_t lddx, float *dw, cudaStream_t stream)
{
    void *scratch = nullptr;
    if (crmsn_status s = scratch_for_current_device(&scratch)) return s;
    if (T > 0) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return CRMSN_ERR_CUDA;
        }
        // 0 means H or the device is invalid; rmsnorm_bwd reports which.
        const size_t need = rmsnorm_bwd_workspace_bytes(T, H, dev, g_residual != nullptr);
        if (need > kScratchBytes) return CRMSN_ERR_SCRATCH_LIMIT;
    }
    return rmsnorm_bwd(g, ldg, x, ldx, w, w_dtype, weight_bias, rstd, g_residual, ldgr, T, H, dx,
                       lddx, dw, scratch, kScratchBytes, stream);
}
