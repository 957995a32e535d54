// launch.h -- parameter blocks and launch entry points shared between the
// host ABI (api.cu) and the kernel translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "common.cuh"

namespace crmsn {

// Largest CTA of the forward kernel (its __launch_bounds__) and of the
// backward kernel.
constexpr int kFwdMaxThreads = 512;
constexpr int kBwdMaxThreads = 512;
// Backward CTAs per SM: at most kBwdMaxCtasPerSm, and at most as many as
// the SM's 228 KB of shared memory can hold at the smallest ring a CTA uses
// (two stages of g and x and the FP32 weight table: 12 bytes per column), so
// the workspace -- one FP32 partial row per CTA -- stays below 12 MB for
// every H on a 152-SM GB300.  (Measured at H = 4096: three or four CTAs per
// SM of a narrower layout were slower than two of 256 threads.)
constexpr int kBwdMaxCtasPerSm = 2;
inline int bwd_max_ctas_per_sm(int64_t H)
{
    const int64_t n = (int64_t)(228 * 1024) / (12 * (H > 0 ? H : 1));
    return n < 1 ? 1 : (n > kBwdMaxCtasPerSm ? kBwdMaxCtasPerSm : (int)n);
}
// Multi-warp row groups of the backward: at most this many per CTA (a group
// has at least 96 threads and a CTA at most 256 threads' worth of groups)
// and at most this many warps each.
constexpr int kBwdMaxGroups = 4;
constexpr int kBwdMaxGroupWarps = kBwdMaxThreads / 32;

enum InKind { IN_PLAIN = 0, IN_RESIDUAL = 1, IN_GATED = 2, IN_LAYERNORM = 3 };
// How the forward holds the weight: WK_MIX, a BF16 weight with no bias, kept
// as packed BF16 and multiplied by h exactly (mixed-precision FMA); WK_BF16
// and WK_F32, the effective weight f32(w + bias) of a BF16 or FP32 weight in
// FP32 registers.
enum WeightKind { WK_MIX = 0, WK_BF16 = 1, WK_F32 = 2 };
enum OutKind {
    OUT_Y = 0,         // y = bf16(o)
    OUT_Q = 1,         // q = fp8(o / scale)
    OUT_BLOCK = 2,     // normed = bf16(o); 1x128 block FP8 + block scales
    OUT_ADA = 3,       // out = bf16(o * (1 + sc) + sh); gate_out copy
    OUT_ADA_Q = 4,     // out = e4m3((o * (1 + sc) + sh) / scale); gate_out copy
    OUT_SILU = 5,      // y = bf16(silu(o))
    OUT_SILU_Q = 6     // q = e4m3(silu(o) / scale), scale 1 when p.scale is NULL
};

struct FwdParams {
    const uint16_t *x;   int64_t ldx;
    const uint16_t *r;   int64_t ldr;     // residual stream (in)
    const uint16_t *gate; int64_t ldgate;
    const void *w;       float bias;      float eps;
    int64_t T;           int H;
    uint16_t *y;         int64_t ldy;     // y / normed / ada out
    uint16_t *hn;        int64_t ldh;     // h_new (may equal r)
    float *rstd;                          // nullable
    uint8_t *q;          int64_t ldq;     // FP8 out
    const float *scale;                   // static FP8 scale (device)
    float *bscale;       int64_t ldT;     // block scales [H/128][ldT]
    const uint16_t *style; int64_t lds;   // style row stride (0: broadcast)
    uint16_t *gate_out;  int64_t ldgo;
    const float *beta;                    // LayerNorm shift [H] (w is gamma)
    float *mean;                          // LayerNorm row means (nullable)
    int tpr;             int rpc;
#ifdef CRMSN_DEBUG
    DebugRanges dbg;                      // the call's tensors (debug build)
#endif
};

struct BwdParams {
    const uint16_t *g;   int64_t ldg;
    const uint16_t *x;   int64_t ldx;
    const void *w;       float bias;
    const float *rstd;
    const uint16_t *gres; int64_t ldgr;
    uint16_t *dx;        int64_t lddx;
    float *part;                          // [nchunk][H] partial dw rows
    float *dw;                            // [H], written by the column CTAs
    int64_t T;           int H;
    int nchunk;          int tpr;         int rpc;
    int ncols;           int colw;        // column form: strips and their width (0: off)
#ifdef CRMSN_DEBUG
    DebugRanges dbg;                      // the call's tensors (debug build)
#endif
};

// Column form of the backward's dw (bwd.cuh): used when T is at most
// kBwdColumnRows.  Strips of colw columns: the widest power of two in
// [16, 256] (16-byte accesses; [16, 64] for 4-byte ones) that still gives at
// least `strips` strips (else 16).  A strip CTA reads 4 bytes per row and
// column, a row CTA 6 per row and column of its chunk, so about 0.4 of the
// resident CTAs should take strips: 128 strips when the layout's CTA (of
// `threads` threads) fits twice on an SM, 64 when it fits once (more than
// 256 threads).  A function of T, H and the layout only, like the sum's
// order.
constexpr int64_t kBwdColumnRows = 2048;
inline int bwd_column_width(int64_t T, int64_t H, int vec, int threads)
{
    if (T > kBwdColumnRows) return 0;
    const int top = vec == 8 ? 256 : 64;
    const int strips = threads > 256 ? 64 : 128;
    int cw = 16;
    while (cw < top && (H + 2 * cw - 1) / (2 * cw) >= strips) cw *= 2;
    return cw;
}

// Row layout picked by the host: VEC elements per access, VPT accesses per
// thread, tpr threads per row (SUB: a power of two <= 32), rpc rows per CTA.
struct Layout {
    int vec, vpt, tpr, rpc;
    bool sub;
};

// Forward launches, one per epilogue family (fwd_*.cu).
// Devices whose dynamic shared-memory opt-in is remembered (beyond them the
// attribute is simply set on every launch that needs it).
constexpr int kOptInDevices = 64;

// Lets kern use `smem` bytes of dynamic shared memory on the current device
// (cudaFuncSetAttribute acts on the current device's context, and the
// default allows 48 KB including the kernel's static shared memory).
// `opted` is the caller's per-kernel record of the largest size set on each
// device, so the attribute is set once per kernel, device and larger size.
// A miss sets the attribute to the larger of the request and the recorded
// size, under one lock with the record update, so two threads asking for
// different sizes can never leave the attribute below the record.
inline std::mutex &opt_in_mutex()
{
    static std::mutex m;
    return m;
}

template <typename Kernel>
cudaError_t opt_in_smem(Kernel kern, size_t smem, std::atomic<int> (&opted)[kOptInDevices])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < kOptInDevices;
    if (!tracked)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if ((int)smem <= opted[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(opt_in_mutex());
    const int cur = opted[dev].load(std::memory_order_relaxed);
    if ((int)smem <= cur) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) opted[dev].store((int)smem, std::memory_order_release);
    return e;
}

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic
// dependent launch allowed: the grid may be scheduled while the kernel before
// it in the stream is still running.  Every kernel of this library that is
// launched this way executes griddepcontrol.wait before its first access to
// global memory, which returns once the preceding grid has completed and its
// writes are visible, so stream order is kept.  Where the attribute is
// refused the launch is an ordinary stream-ordered one (the wait then
// returns at once).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kern, args...);
    }
    return e;
}

cudaError_t launch_fwd_y(const FwdParams &p, int in, int wk, const Layout &L, cudaStream_t s);
cudaError_t launch_fwd_q(const FwdParams &p, int in, int wk, int fp8k, const Layout &L, cudaStream_t s);
cudaError_t launch_fwd_block(const FwdParams &p, const Layout &L, cudaStream_t s);
cudaError_t launch_fwd_ada(const FwdParams &p, bool gated_fp8, const Layout &L, cudaStream_t s);
// RMSNorm + SiLU (BF16, or E4M3 when fp8) and LayerNorm (BF16 when
// fp8k < 0, else FP8 of that kind), fwd_silu_ln.cu.
cudaError_t launch_fwd_silu(const FwdParams &p, int wk, bool fp8, const Layout &L, cudaStream_t s);
cudaError_t launch_fwd_layernorm(const FwdParams &p, int fp8k, const Layout &L, cudaStream_t s);

// Backward (bwd.cu).
// Picks the chunk count (resident CTAs per SM x sms, at most
// kBwdMaxCtasPerSm x sms and at most one per row group), launches the dx /
// partial-dw kernel and then the fixed-order dw reduction (bwd_reduce.cu);
// with p.ncols > 0 (the column form) one launch writes dx and dw.
cudaError_t launch_bwd(BwdParams p, bool w32, bool gres, const Layout &L, int sms, float *dw,
                       cudaStream_t s);
// The dx / partial-dw kernel alone, per weight type and g_residual
// (bwd_bf16w.cu, bwd_bf16w_gres.cu, bwd_f32w.cu, bwd_f32w_gres.cu, compiled
// in parallel); *nchunk receives the chunk count it used.
cudaError_t launch_bwd_bf16w_plain(const BwdParams &p, const Layout &L, int sms, int *nchunk, cudaStream_t s);
cudaError_t launch_bwd_bf16w_gres(const BwdParams &p, const Layout &L, int sms, int *nchunk, cudaStream_t s);
cudaError_t launch_bwd_f32w_plain(const BwdParams &p, const Layout &L, int sms, int *nchunk, cudaStream_t s);
cudaError_t launch_bwd_f32w_gres(const BwdParams &p, const Layout &L, int sms, int *nchunk, cudaStream_t s);

}  // namespace crmsn
