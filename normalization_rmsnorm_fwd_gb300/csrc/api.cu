// api.cu -- the C ABI declared in include/crmsnorm.h: argument checks,
// row-layout choice and kernel dispatch.  Nothing here allocates or
// synchronises; every check happens before the first launch.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "crmsnorm.h"
#include "launch.h"

using namespace crmsn;

namespace {

// ------------------------------------------------------------ device info --

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------ layouts ----

int next_pow2(int v)
{
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Forward: rows of <= 64 vectors use a sub-warp group (two vectors per thread
// at most); wider rows use a group of whole warps, at most 16, holding 2 or 4
// 16-byte vectors (2..16 4-byte vectors) per thread, choosing the fewest idle
// lanes (ties: the first preference).  The Ada epilogues stream three more
// tensors per element and prefer fewer vectors per thread (narrow).  Narrow
// groups share a CTA so that CTAs have about 256 threads.  need16: the 1x128 block epilogue needs
// 16-lane aligned groups.
Layout choose_fwd(int H, int vec, bool need16, bool narrow)
{
    const int nvec = H / vec;
    Layout L{};
    L.vec = vec;
    if (nvec <= 64) {
        int tpr = next_pow2((nvec + 1) / 2);
        if (need16 && tpr < 16) tpr = 16;
        if (tpr > 32) tpr = 32;
        L.tpr = tpr;
        L.vpt = (nvec + tpr - 1) / tpr;
        L.sub = true;
        L.rpc = 256 / tpr;
        return L;
    }
    static const int prefs8[] = {4, 2}, prefs8_narrow[] = {2, 4};
    static const int prefs2[] = {16, 8, 4, 2}, prefs2_narrow[] = {8, 4, 16, 2};
    const int *prefs = vec == 8 ? (narrow ? prefs8_narrow : prefs8)
                                : (narrow ? prefs2_narrow : prefs2);
    const int np = vec == 8 ? 2 : 4;
    int best = -1;
    long best_waste = 0;
    for (int i = 0; i < np; ++i) {
        const int vpt = prefs[i];
        const int nw = (nvec + 32 * vpt - 1) / (32 * vpt);
        if (nw > kFwdMaxThreads / 32) continue;
        const long waste = (long)nw * 32 * vpt - nvec;
        if (best < 0 || waste < best_waste) {
            best = vpt;
            best_waste = waste;
        }
    }
    L.vpt = best;
    L.tpr = 32 * ((nvec + 32 * best - 1) / (32 * best));
    L.sub = false;
    L.rpc = L.tpr >= 256 ? 1 : 256 / L.tpr;
    return L;
}

// Backward: groups of at most 8 warps while a thread holds at most 16
// elements (2 16-byte vectors), so that a row's cross-thread reduction stays
// short and two CTAs fit per SM; wider rows grow to 16 warps, then to more
// vectors per thread.  The cp.async ring keeps the next rows in flight.
// (Measured at H = 4096: 32 elements per thread in 128-thread CTAs, three
// per SM, took 84.7 us against 72.3 us.)
Layout choose_bwd(int H, int vec)
{
    const int nvec = H / vec;
    Layout L{};
    L.vec = vec;
    if (nvec <= 64) {
        int tpr = next_pow2((nvec + 1) / 2);
        if (tpr > 32) tpr = 32;
        L.tpr = tpr;
        L.vpt = (nvec + tpr - 1) / tpr;
        L.sub = true;
        L.rpc = 256 / tpr;
        return L;
    }
    auto nw = [&](int vpt) { return (nvec + 32 * vpt - 1) / (32 * vpt); };
    int vpt = 1;
    while (nw(vpt) > 8 && vpt * vec < 16) vpt *= 2;
    while (nw(vpt) > kBwdMaxThreads / 32) vpt *= 2;
    L.vpt = vpt;
    L.tpr = 32 * nw(vpt);
    L.sub = false;
    L.rpc = L.tpr >= 256 ? 1 : 256 / L.tpr;
    return L;
}

// ------------------------------------------------------------ checks -----

bool al(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// A row-strided 2-D region: rows x cols elements of es bytes, row stride ld.
struct Region {
    const void *p;
    int64_t rows, ld, cols;
    int es;
};

bool same_tensor(const Region &a, const Region &b)
{
    return a.p == b.p && a.es == b.es && a.cols == b.cols && (a.rows <= 1 || a.ld == b.ld);
}

// True when two regions may share a byte.  Regions with the same row period
// whose column ranges do not meet inside the period (interleaved slices of
// one buffer) are disjoint.
bool overlaps(const Region &a, const Region &b)
{
    if (!a.p || !b.p || a.rows == 0 || b.rows == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    const uintptr_t a1 = a0 + (uintptr_t)(((a.rows - 1) * a.ld + a.cols) * a.es);
    const uintptr_t b1 = b0 + (uintptr_t)(((b.rows - 1) * b.ld + b.cols) * b.es);
    if (a1 <= b0 || b1 <= a0) return false;
    const int64_t pa = a.ld * a.es, pb = b.ld * b.es;
    if (a.rows > 1 && b.rows > 1 && pa == pb && pa > 0) {
        const int64_t d = (int64_t)(b0 - a0);
        int64_t off = d % pa;
        if (off < 0) off += pa;
        const int64_t wa = a.cols * a.es, wb = b.cols * b.es;
        if (off >= wa && off + wb <= pa) return false;
    }
    return true;
}

// Every output must be disjoint from every other tensor, except for the one
// input it may replace in place (same pointer and stride).
struct Tensor {
    Region r;
    bool out;
    int may_replace;   // index of the input it may equal, or -1
};

crmsn_status check_alias(const Tensor *ts, int n)
{
    for (int i = 0; i < n; ++i) {
        if (!ts[i].out || !ts[i].r.p) continue;
        for (int j = 0; j < n; ++j) {
            if (j == i || !ts[j].r.p) continue;
            if (ts[i].may_replace == j && same_tensor(ts[i].r, ts[j].r)) continue;
            if (ts[j].out && ts[j].may_replace == i && same_tensor(ts[i].r, ts[j].r)) continue;
            if (overlaps(ts[i].r, ts[j].r)) return CRMSN_ERR_ALIAS;
        }
    }
    return CRMSN_OK;
}

// Vector width for a set of BF16 row tensors, FP8 row tensors and the weight:
// 8 when every base is 16-byte aligned (FP8: 8-byte) and every stride and H
// are multiples of 8; 2 when bases are 4-byte (FP8: 2-byte) aligned and
// strides even; 0 otherwise.
struct Access {
    const void *p;
    int64_t ld;
    int kind;   // 0 = BF16 rows, 1 = FP8 rows, 2 = BF16 vector, 3 = FP32 vector
};

int pick_vec(const Access *a, int n, int64_t H, int64_t T)
{
    auto fits = [&](int vec) {
        if (H % vec) return false;
        for (int i = 0; i < n; ++i) {
            if (!a[i].p) continue;
            uintptr_t need;
            switch (a[i].kind) {
                case 0: case 2: need = 2 * vec; break;
                case 1: need = vec; break;
                default: need = 4 * (vec == 8 ? 4 : 2); break;
            }
            if (!al(a[i].p, need)) return false;
            if ((a[i].kind == 0 || a[i].kind == 1) && T > 1 && a[i].ld % vec) return false;
        }
        return true;
    };
    if (fits(8)) return 8;
    if (fits(2)) return 2;
    return 0;
}

bool bad_float(float v) { return !std::isfinite(v); }

// How the forward holds the weight (launch.h WeightKind): a BF16 weight with
// no bias stays packed (its products with h are exact), anything else is
// turned into the FP32 effective weight once.
int weight_kind(int w_dtype, float weight_bias)
{
    if (w_dtype == CRMSN_F32) return WK_F32;
    return weight_bias == 0.f ? WK_MIX : WK_BF16;
}

crmsn_status launched(cudaError_t e)
{
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return CRMSN_ERR_CUDA;
    }
    return CRMSN_OK;
}

crmsn_status check_h(int64_t H)
{
    if (H < 1) return CRMSN_ERR_SHAPE;
    if (H > CRMSN_MAX_H || (H & 1)) return CRMSN_ERR_UNSUPPORTED_H;
    return CRMSN_OK;
}

constexpr int64_t kMaxBlocks = 0x7fffffff;

#ifdef CRMSN_DEBUG
// The debug build's violation word (one per device; its address is looked up
// once per device) and the range table of a call: every tensor of the call,
// the outputs writable.
__device__ unsigned long long g_debug_word;
constexpr int kDebugDevices = 64;
std::mutex g_debug_mutex;
unsigned long long *g_debug_word_ptr[kDebugDevices];

unsigned long long *debug_word()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDebugDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_debug_mutex);
    if (!g_debug_word_ptr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_debug_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_debug_word_ptr[dev] = static_cast<unsigned long long *>(a);
    }
    return g_debug_word_ptr[dev];
}

template <int N>
DebugRanges debug_ranges(const Tensor (&ts)[N])
{
    static_assert(N <= kDebugMaxRanges, "more tensors than debug ranges");
    DebugRanges d{};
    d.word = debug_word();
    for (int i = 0; i < N; ++i) {
        const Region &r = ts[i].r;
        if (!r.p || r.rows == 0) continue;
        const uintptr_t a = (uintptr_t)r.p;
        d.lo[d.n] = a;
        d.hi[d.n] = a + (uintptr_t)(((r.rows - 1) * r.ld + r.cols) * r.es);
        if (ts[i].out) d.writable |= 1u << d.n;
        ++d.n;
    }
    // Self-test of the guard: CRMSN_DEBUG_TRIM_OUTPUT=k takes k bytes off
    // the end of the first output's range (the guard's view only: the
    // buffer itself is untouched), so the stores there are reported and
    // skipped.
    if (const char *t = getenv("CRMSN_DEBUG_TRIM_OUTPUT")) {
        const unsigned long long k = strtoull(t, nullptr, 10);
        for (int i = 0; i < d.n; ++i)
            if ((d.writable >> i) & 1u) {
                d.hi[i] = d.hi[i] - k > d.lo[i] ? d.hi[i] - k : d.lo[i];
                break;
            }
    }
    return d;
}
#define CRMSN_SET_DEBUG(p, ts) ((p).dbg = debug_ranges(ts))
#else
#define CRMSN_SET_DEBUG(p, ts) ((void)0)
#endif

}  // namespace

// ======================================================================
extern "C" {

const char *crmsn_status_str(crmsn_status s)
{
    switch (s) {
        case CRMSN_OK: return "ok";
        case CRMSN_ERR_NULL: return "a required pointer is NULL";
        case CRMSN_ERR_SHAPE: return "invalid shape or row stride";
        case CRMSN_ERR_UNSUPPORTED_H: return "hidden size not supported by this operation";
        case CRMSN_ERR_ALIGNMENT: return "pointer or row stride misaligned";
        case CRMSN_ERR_DTYPE: return "unknown weight dtype or FP8 kind";
        case CRMSN_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case CRMSN_ERR_ALIAS: return "an output overlaps another tensor";
        case CRMSN_ERR_CUDA: return "CUDA runtime error";
        case CRMSN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case CRMSN_ERR_ARG: return "eps or scale out of range";
        case CRMSN_ERR_SCRATCH_LIMIT: return "problem needs more than the built-in 16 MiB backward scratch";
        case CRMSN_ERR_NOT_DEBUG_BUILD: return "this library was built without the debug bounds guard";
    }
    return "unknown status";
}

crmsn_status crmsn_debug_status(uint64_t *violation)
{
    if (!violation) return CRMSN_ERR_NULL;
    *violation = 0;
#ifdef CRMSN_DEBUG
    if (!debug_word()) return CRMSN_ERR_CUDA;
    unsigned long long w = 0;
    const unsigned long long zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&w, g_debug_word, sizeof w) != cudaSuccess ||
        cudaMemcpyToSymbol(g_debug_word, &zero, sizeof zero) != cudaSuccess) {
        (void)cudaGetLastError();
        return CRMSN_ERR_CUDA;
    }
    *violation = w;
    return CRMSN_OK;
#else
    return CRMSN_ERR_NOT_DEBUG_BUILD;
#endif
}

crmsn_status rmsnorm_supports(int64_t H, int w_dtype, int op)
{
    if (w_dtype != CRMSN_BF16 && w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
    switch (op) {
        case CRMSN_OP_FWD:
        case CRMSN_OP_BWD:
        case CRMSN_OP_QUANT:
            return check_h(H);
        case CRMSN_OP_BLOCK_QUANT:
            if (w_dtype != CRMSN_BF16) return CRMSN_ERR_DTYPE;
            if (H < 1) return CRMSN_ERR_SHAPE;
            return (H % 128 || H > CRMSN_MAX_H) ? CRMSN_ERR_UNSUPPORTED_H : CRMSN_OK;
        case CRMSN_OP_SILU:
            return check_h(H);
        case CRMSN_OP_LAYERNORM:
            if (w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
            return check_h(H);
        case CRMSN_OP_ADA_STYLE:
        case CRMSN_OP_GATED_ADA_FP8:
            if (w_dtype != CRMSN_BF16) return CRMSN_ERR_DTYPE;
            if (H < 1 || (H & 1)) return CRMSN_ERR_SHAPE;
            return H > CRMSN_MAX_H ? CRMSN_ERR_UNSUPPORTED_H : CRMSN_OK;
        default:
            return CRMSN_ERR_ARG;
    }
}

crmsn_status rmsnorm_fwd(const void *x, int64_t ldx, const void *residual, int64_t ldr,
                         const void *w, int w_dtype, float weight_bias, float eps,
                         int64_t T, int64_t H, void *y, int64_t ldy, float *rstd,
                         void *h_new, int64_t ldh, cudaStream_t stream)
{
    if (T < 0) return CRMSN_ERR_SHAPE;
    if (crmsn_status s = check_h(H)) return s;
    if (w_dtype != CRMSN_BF16 && w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
    if (bad_float(eps) || eps < 0.f || bad_float(weight_bias)) return CRMSN_ERR_ARG;
    if (T == 0) return CRMSN_OK;
    if (!x || !w || !y || (residual && !h_new)) return CRMSN_ERR_NULL;
    if (T > 1 && (ldx < H || ldy < H || (residual && (ldr < H || ldh < H)))) return CRMSN_ERR_SHAPE;
    const int wes = w_dtype == CRMSN_F32 ? 4 : 2;
    const bool res = residual != nullptr;
    const Tensor ts[] = {
        {{x, T, ldx, H, 2}, false, -1},
        {{residual, T, ldr, H, 2}, false, -1},
        {{w, 1, H, H, wes}, false, -1},
        {{y, T, ldy, H, 2}, true, 0},
        {{res ? h_new : nullptr, T, ldh, H, 2}, true, 1},
        {{rstd, 1, T, T, 4}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 6)) return s;
    const Access acc[] = {{x, ldx, 0}, {residual, ldr, 0}, {y, ldy, 0},
                          {res ? h_new : nullptr, ldh, 0}, {w, 0, w_dtype == CRMSN_F32 ? 3 : 2}};
    const int vec = pick_vec(acc, 5, H, T);
    if (!vec || (rstd && !al(rstd, 4))) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_fwd((int)H, vec, false, false);
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.r = static_cast<const uint16_t *>(residual); p.ldr = ldr;
    p.w = w; p.bias = weight_bias; p.eps = eps;
    p.T = T; p.H = (int)H;
    p.y = static_cast<uint16_t *>(y); p.ldy = ldy;
    p.hn = static_cast<uint16_t *>(h_new); p.ldh = ldh;
    p.rstd = rstd;
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_y(p, res ? IN_RESIDUAL : IN_PLAIN, weight_kind(w_dtype, weight_bias), L,
                                 stream));
}

size_t rmsnorm_bwd_workspace_bytes(int64_t rows, int64_t H, int device, int residual)
{
    (void)rows;
    (void)residual;
    if (check_h(H) != CRMSN_OK) return 0;
    const int sms = sm_count(device);
    if (sms <= 0) return 0;
    return align_up((size_t)bwd_max_ctas_per_sm(H) * sms * (size_t)H * sizeof(float), 256) + 256;
}

crmsn_status rmsnorm_bwd(const void *g, int64_t ldg, const void *x, int64_t ldx,
                         const void *w, int w_dtype, float weight_bias, const float *rstd,
                         const void *g_residual, int64_t ldgr, int64_t T, int64_t H,
                         void *dx, int64_t lddx, float *dw, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream)
{
    if (T < 0) return CRMSN_ERR_SHAPE;
    if (crmsn_status s = check_h(H)) return s;
    if (w_dtype != CRMSN_BF16 && w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
    if (bad_float(weight_bias)) return CRMSN_ERR_ARG;
    if (!dw) return CRMSN_ERR_NULL;
    if (T == 0) {
        if (!al(dw, 4)) return CRMSN_ERR_ALIGNMENT;
        return launched(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), stream));
    }
    if (!g || !x || !w || !rstd || !dx || !workspace) return CRMSN_ERR_NULL;
    if (T > 1 && (ldg < H || ldx < H || lddx < H || (g_residual && ldgr < H))) return CRMSN_ERR_SHAPE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return launched(cudaErrorNoDevice);
    const size_t need = rmsnorm_bwd_workspace_bytes(T, H, dev, g_residual != nullptr);
    if (need == 0) return CRMSN_ERR_CUDA;
    if (!al(workspace, 256) || workspace_bytes < need) return CRMSN_ERR_WORKSPACE;
    const int wes = w_dtype == CRMSN_F32 ? 4 : 2;
    const Tensor ts[] = {
        {{g, T, ldg, H, 2}, false, -1},
        {{x, T, ldx, H, 2}, false, -1},
        {{w, 1, H, H, wes}, false, -1},
        {{rstd, 1, T, T, 4}, false, -1},
        {{g_residual, T, ldgr, H, 2}, false, -1},
        {{dx, T, lddx, H, 2}, true, 0},
        {{dw, 1, H, H, 4}, true, -1},
        {{workspace, 1, (int64_t)workspace_bytes, (int64_t)workspace_bytes, 1}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 8)) return s;
    if (!al(dw, 4) || !al(rstd, 4)) return CRMSN_ERR_ALIGNMENT;
    const Access acc[] = {{g, ldg, 0}, {x, ldx, 0}, {dx, lddx, 0}, {g_residual, ldgr, 0},
                          {w, 0, w_dtype == CRMSN_F32 ? 3 : 2}};
    const int vec = pick_vec(acc, 5, H, T);
    if (!vec) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_bwd((int)H, vec);

    BwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.g = static_cast<const uint16_t *>(g); p.ldg = ldg;
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.w = w; p.bias = weight_bias; p.rstd = rstd;
    p.gres = static_cast<const uint16_t *>(g_residual); p.ldgr = ldgr;
    p.dx = static_cast<uint16_t *>(dx); p.lddx = lddx;
    p.part = static_cast<float *>(workspace);
    p.dw = dw;
    p.T = T; p.H = (int)H; p.tpr = L.tpr; p.rpc = L.rpc;
    p.colw = bwd_column_width(T, H, vec, L.tpr * L.rpc);
    p.ncols = p.colw > 0 ? (int)((H + p.colw - 1) / p.colw) : 0;
    return launched(launch_bwd(p, w_dtype == CRMSN_F32, g_residual != nullptr, L, sm_count(dev),
                               dw, stream));
}

crmsn_status fused_add_rmsnorm_quant(void *out, int64_t ldo, int fp8_kind, const void *x,
                                     int64_t ldx, void *residual, int64_t ldr, const void *w,
                                     int w_dtype, float weight_bias, const float *scale,
                                     float eps, int64_t T, int64_t H, float *rstd,
                                     cudaStream_t stream)
{
    if (T < 0) return CRMSN_ERR_SHAPE;
    if (crmsn_status s = check_h(H)) return s;
    if (w_dtype != CRMSN_BF16 && w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
    if (fp8_kind != CRMSN_E4M3 && fp8_kind != CRMSN_E5M2) return CRMSN_ERR_DTYPE;
    if (bad_float(eps) || eps < 0.f || bad_float(weight_bias)) return CRMSN_ERR_ARG;
    if (T == 0) return CRMSN_OK;
    if (!out || !x || !w || !scale) return CRMSN_ERR_NULL;
    if (T > 1 && (ldo < H || ldx < H || (residual && ldr < H))) return CRMSN_ERR_SHAPE;
    const int wes = w_dtype == CRMSN_F32 ? 4 : 2;
    const Tensor ts[] = {
        {{x, T, ldx, H, 2}, false, -1},
        {{w, 1, H, H, wes}, false, -1},
        {{scale, 1, 1, 1, 4}, false, -1},
        {{residual, T, ldr, H, 2}, true, -1},   // updated in place
        {{out, T, ldo, H, 1}, true, -1},
        {{rstd, 1, T, T, 4}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 6)) return s;
    const Access acc[] = {{x, ldx, 0}, {residual, ldr, 0}, {out, ldo, 1},
                          {w, 0, w_dtype == CRMSN_F32 ? 3 : 2}};
    const int vec = pick_vec(acc, 4, H, T);
    if (!vec || !al(scale, 4) || (rstd && !al(rstd, 4))) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_fwd((int)H, vec, false, false);
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.r = static_cast<const uint16_t *>(residual); p.ldr = ldr;
    p.w = w; p.bias = weight_bias; p.eps = eps;
    p.T = T; p.H = (int)H;
    p.hn = static_cast<uint16_t *>(residual); p.ldh = ldr;
    p.rstd = rstd;
    p.q = static_cast<uint8_t *>(out); p.ldq = ldo;
    p.scale = scale;
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_q(p, residual ? IN_RESIDUAL : IN_PLAIN,
                                 weight_kind(w_dtype, weight_bias), fp8_kind, L, stream));
}

crmsn_status fused_add_rmsnorm_fp8_block_quant(void *out, float *block_scale, int64_t ldT,
                                               void *normed_out, const void *x, int64_t ldx,
                                               void *residual, int64_t ldr, const void *w,
                                               float eps, int64_t T, int64_t H,
                                               cudaStream_t stream)
{
    if (T < 0 || H < 1) return CRMSN_ERR_SHAPE;
    if (H % 128 || H > CRMSN_MAX_H) return CRMSN_ERR_UNSUPPORTED_H;
    if (bad_float(eps) || eps < 0.f) return CRMSN_ERR_ARG;
    if (ldT < T) return CRMSN_ERR_SHAPE;
    if (T == 0) return CRMSN_OK;
    if (!out || !block_scale || !normed_out || !x || !residual || !w) return CRMSN_ERR_NULL;
    if (T > 1 && (ldx < H || ldr < H)) return CRMSN_ERR_SHAPE;
    const Tensor ts[] = {
        {{x, T, ldx, H, 2}, false, -1},
        {{w, 1, H, H, 2}, false, -1},
        {{residual, T, ldr, H, 2}, true, -1},
        {{out, T, H, H, 1}, true, -1},
        {{normed_out, T, H, H, 2}, true, -1},
        {{block_scale, H / 128, ldT, T, 4}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 6)) return s;
    const Access acc[] = {{x, ldx, 0}, {residual, ldr, 0}, {normed_out, H, 0}, {out, H, 1},
                          {w, 0, 2}};
    if (pick_vec(acc, 5, H, T) != 8 || !al(block_scale, 4)) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_fwd((int)H, 8, true, false);
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.r = static_cast<const uint16_t *>(residual); p.ldr = ldr;
    p.w = w; p.bias = 0.f; p.eps = eps;
    p.T = T; p.H = (int)H;
    p.y = static_cast<uint16_t *>(normed_out); p.ldy = H;
    p.hn = static_cast<uint16_t *>(residual); p.ldh = ldr;
    p.q = static_cast<uint8_t *>(out); p.ldq = H;
    p.bscale = block_scale; p.ldT = ldT;
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_block(p, L, stream));
}

static crmsn_status ada_common(void *residual, const void *x, const void *gate, const void *w,
                               const void *style, int64_t style_rows, const float *scale,
                               float eps, int64_t T, int64_t D, void *out, void *gate_out,
                               bool gated, cudaStream_t stream)
{
    if (T < 0 || D < 1 || (D & 1)) return CRMSN_ERR_SHAPE;
    if (D > CRMSN_MAX_H) return CRMSN_ERR_UNSUPPORTED_H;
    if (bad_float(eps) || eps < 0.f) return CRMSN_ERR_ARG;
    if (T == 0) return CRMSN_OK;
    if (!x || !w || !style || !out || !gate_out) return CRMSN_ERR_NULL;
    if (gated && (!residual || !gate || !scale)) return CRMSN_ERR_NULL;
    if (style_rows != 1 && style_rows != T) return CRMSN_ERR_SHAPE;
    const int oes = gated ? 1 : 2;
    const Tensor ts[] = {
        {{x, T, D, D, 2}, false, -1},
        {{gated ? gate : nullptr, T, D, D, 2}, false, -1},
        {{w, 1, D, D, 2}, false, -1},
        {{style, style_rows, 3 * D, 3 * D, 2}, false, -1},
        {{gated ? scale : nullptr, 1, 1, 1, 4}, false, -1},
        {{gated ? residual : nullptr, T, D, D, 2}, true, -1},
        {{out, T, D, D, oes}, true, -1},
        {{gate_out, T, D, D, 2}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 8)) return s;
    const Access acc[] = {{x, D, 0}, {gated ? gate : nullptr, D, 0},
                          {gated ? residual : nullptr, D, 0}, {style, 3 * D, 0},
                          {out, D, gated ? 1 : 0}, {gate_out, D, 0}, {w, 0, 2}};
    const int vec = pick_vec(acc, 7, D, T > 1 ? T : 2);
    if (!vec || (gated && !al(scale, 4))) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_fwd((int)D, vec, false, true);
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = D;
    p.r = static_cast<const uint16_t *>(residual); p.ldr = D;
    p.gate = static_cast<const uint16_t *>(gate); p.ldgate = D;
    p.w = w; p.bias = 0.f; p.eps = eps;
    p.T = T; p.H = (int)D;
    p.y = static_cast<uint16_t *>(out); p.ldy = D;
    p.hn = static_cast<uint16_t *>(residual); p.ldh = D;
    p.q = static_cast<uint8_t *>(out); p.ldq = D;
    p.scale = scale;
    p.style = static_cast<const uint16_t *>(style); p.lds = style_rows == 1 ? 0 : 3 * D;
    p.gate_out = static_cast<uint16_t *>(gate_out); p.ldgo = D;
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_ada(p, gated, L, stream));
}

crmsn_status ada_rms_norm_style(const void *x, const void *w, const void *style,
                                int64_t style_rows, float eps, int64_t T, int64_t D, void *out,
                                void *gate_out, cudaStream_t stream)
{
    return ada_common(nullptr, x, nullptr, w, style, style_rows, nullptr, eps, T, D, out,
                      gate_out, false, stream);
}

crmsn_status gate_residual_ada_norm_fp8(void *residual, const void *x, const void *gate,
                                        const void *w, const void *style, int64_t style_rows,
                                        const float *scale, float eps, int64_t T, int64_t D,
                                        void *out, void *gate_out, cudaStream_t stream)
{
    return ada_common(residual, x, gate, w, style, style_rows, scale, eps, T, D, out, gate_out,
                      true, stream);
}

crmsn_status fused_rmsnorm_silu(void *out, int64_t ldo, int out_format, const void *x,
                                int64_t ldx, const void *w, int w_dtype, float weight_bias,
                                const float *scale, float eps, int64_t T, int64_t H,
                                float *rstd, cudaStream_t stream)
{
    if (T < 0) return CRMSN_ERR_SHAPE;
    if (crmsn_status s = check_h(H)) return s;
    if (w_dtype != CRMSN_BF16 && w_dtype != CRMSN_F32) return CRMSN_ERR_DTYPE;
    if (out_format != CRMSN_OUT_BF16 && out_format != CRMSN_OUT_E4M3) return CRMSN_ERR_DTYPE;
    if (bad_float(eps) || eps < 0.f || bad_float(weight_bias)) return CRMSN_ERR_ARG;
    if (T == 0) return CRMSN_OK;
    if (!out || !x || !w) return CRMSN_ERR_NULL;
    if (T > 1 && (ldo < H || ldx < H)) return CRMSN_ERR_SHAPE;
    const bool fp8 = out_format == CRMSN_OUT_E4M3;
    const int wes = w_dtype == CRMSN_F32 ? 4 : 2;
    const Tensor ts[] = {
        {{x, T, ldx, H, 2}, false, -1},
        {{w, 1, H, H, wes}, false, -1},
        {{fp8 ? scale : nullptr, 1, 1, 1, 4}, false, -1},
        {{out, T, ldo, H, fp8 ? 1 : 2}, true, fp8 ? -1 : 0},   // BF16 out may replace x
        {{rstd, 1, T, T, 4}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 5)) return s;
    const Access acc[] = {{x, ldx, 0}, {out, ldo, fp8 ? 1 : 0},
                          {w, 0, w_dtype == CRMSN_F32 ? 3 : 2}};
    const int vec = pick_vec(acc, 3, H, T);
    if (!vec || (fp8 && scale && !al(scale, 4)) || (rstd && !al(rstd, 4))) return CRMSN_ERR_ALIGNMENT;
    const Layout L = choose_fwd((int)H, vec, false, false);
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.w = w; p.bias = weight_bias; p.eps = eps;
    p.T = T; p.H = (int)H;
    p.rstd = rstd;
    if (fp8) {
        p.q = static_cast<uint8_t *>(out); p.ldq = ldo;
        p.scale = scale;
    } else {
        p.y = static_cast<uint16_t *>(out); p.ldy = ldo;
    }
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_silu(p, weight_kind(w_dtype, weight_bias), fp8, L, stream));
}

}  // extern "C"

namespace {

// layernorm (fp8k < 0, BF16 out) and layernorm_quant (fp8k = FP8 kind).
crmsn_status layernorm_common(void *out, int64_t ldo, int fp8k, const void *x, int64_t ldx,
                              const float *gamma, const float *beta, const float *scale,
                              float eps, int64_t T, int64_t H, float *mean, float *rstd,
                              cudaStream_t stream)
{
    if (T < 0) return CRMSN_ERR_SHAPE;
    if (crmsn_status s = check_h(H)) return s;
    if (bad_float(eps) || eps < 0.f) return CRMSN_ERR_ARG;
    if (T == 0) return CRMSN_OK;
    const bool fp8 = fp8k >= 0;
    if (!out || !x || !gamma || !beta || (fp8 && !scale)) return CRMSN_ERR_NULL;
    if (T > 1 && (ldo < H || ldx < H)) return CRMSN_ERR_SHAPE;
    const Tensor ts[] = {
        {{x, T, ldx, H, 2}, false, -1},
        {{gamma, 1, H, H, 4}, false, -1},
        {{beta, 1, H, H, 4}, false, -1},
        {{fp8 ? scale : nullptr, 1, 1, 1, 4}, false, -1},
        {{out, T, ldo, H, fp8 ? 1 : 2}, true, fp8 ? -1 : 0},   // BF16 out may replace x
        {{mean, 1, T, T, 4}, true, -1},
        {{rstd, 1, T, T, 4}, true, -1},
    };
    if (crmsn_status s = check_alias(ts, 7)) return s;
    const Access acc[] = {{x, ldx, 0}, {out, ldo, fp8 ? 1 : 0}, {gamma, 0, 3}, {beta, 0, 3}};
    const int vec = pick_vec(acc, 4, H, T);
    if (!vec || (fp8 && !al(scale, 4)) || (mean && !al(mean, 4)) || (rstd && !al(rstd, 4)))
        return CRMSN_ERR_ALIGNMENT;
    Layout L = choose_fwd((int)H, vec, false, false);
    // BF16 output at H = 4096 and 8192: 64 elements per thread (two warps a
    // row at H = 4096), the next row prefetched into L2 only (measured at
    // T * H = 2^26: 49.4 -> 46.5 us and 52.6 -> 48.1 us; the FP8 outputs
    // lost 2-4 % with it and keep 32 elements per thread).
    if (!fp8 && vec == 8 && H % 4096 == 0 && H <= 8192) {
        L.vpt = 8;
        L.tpr = (int)(H / 64);
        L.rpc = L.tpr >= 256 ? 1 : 256 / L.tpr;
    }
    if ((T + L.rpc - 1) / L.rpc > kMaxBlocks) return CRMSN_ERR_SHAPE;

    FwdParams p{};
    CRMSN_SET_DEBUG(p, ts);
    p.x = static_cast<const uint16_t *>(x); p.ldx = ldx;
    p.w = gamma; p.beta = beta; p.eps = eps;
    p.T = T; p.H = (int)H;
    p.rstd = rstd; p.mean = mean;
    if (fp8) {
        p.q = static_cast<uint8_t *>(out); p.ldq = ldo;
        p.scale = scale;
    } else {
        p.y = static_cast<uint16_t *>(out); p.ldy = ldo;
    }
    p.tpr = L.tpr; p.rpc = L.rpc;
    return launched(launch_fwd_layernorm(p, fp8k, L, stream));
}

}  // namespace

extern "C" {

crmsn_status layernorm(void *y, int64_t ldy, const void *x, int64_t ldx, const float *gamma,
                       const float *beta, float eps, int64_t T, int64_t H, float *mean,
                       float *rstd, cudaStream_t stream)
{
    return layernorm_common(y, ldy, -1, x, ldx, gamma, beta, nullptr, eps, T, H, mean, rstd,
                            stream);
}

crmsn_status layernorm_quant(void *out, int64_t ldo, int fp8_kind, const void *x, int64_t ldx,
                             const float *gamma, const float *beta, const float *scale,
                             float eps, int64_t T, int64_t H, float *mean, float *rstd,
                             cudaStream_t stream)
{
    if (fp8_kind != CRMSN_E4M3 && fp8_kind != CRMSN_E5M2) return CRMSN_ERR_DTYPE;
    return layernorm_common(out, ldo, fp8_kind, x, ldx, gamma, beta, scale, eps, T, H, mean,
                            rstd, stream);
}

}  // extern "C"
