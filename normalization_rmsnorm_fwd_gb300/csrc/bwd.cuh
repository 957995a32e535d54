// bwd.cuh -- RMSNorm backward: dx per row and a deterministic FP32 dw.
//
// Source: "FlashInfer normalization operator guide" 6.1-6.3 and the
// "cake_rmsnorm_det_train_forward" Notes:
//   m    = mean(g * w * x)
//   dx   = bf16(rstd*g*w - x*rstd^3*m (+ g_residual))
//   dw   = sum_t g * x * rstd, bitwise reproducible for a given T and SM count.
//
// Design (GB300).  CTA c owns the contiguous row chunk [c*T/n, (c+1)*T/n) of
// a fixed chunk table (n = chunks, a function of T and the SM count).  Each
// thread owns the same columns in every row and keeps, per column, a plain
// FP32 sum (one fused multiply-add per row) of its last kDwBlock rows plus a
// compensated (TwoSum) FP32 pair into which each block sum is folded, all in
// registers, while it walks its chunk (error <= kDwBlock ulp of the summed
// magnitudes).  Elementwise arithmetic uses packed FP32x2 instructions, and
// the products g*x come exact from mixed-precision BF16 FMAs.  Rows stream
// through a ring of shared-memory stages filled with cp.async: every thread
// copies exactly the 16-byte (or 4-byte) pieces of g and x (g_residual) that
// it will itself consume, D rows ahead, and waits only on its own copy groups
// (cp.async.wait_group), so D rows per CTA are in flight without any register
// cost, cross-thread handoff or flag spinning; rstd is read 32 rows at a time
// into registers and broadcast by shuffles.  Multi-warp rows run a software
// pipeline (row i+1's sum formed while row i gets its dx, one CTA barrier per
// row); the per-row integer work is kept to running pointers and counters,
// since at about 20 instructions per element the kernel is bound by issue.
// D is 3, 2 or 1 rows: the deepest ring that fits the shared-memory budget.
// At the end the CTA adds its row groups in group order, column-parallel
// across its threads, and writes one FP32 partial row; a second kernel
// (bwd_reduce.cu) adds the partial rows of each column in a fixed order.
// Both grids are launched with programmatic dependent launch and wait for
// the preceding grid before touching global memory.
//
// Short inputs (the column form, the pages' "column task" for small T): the
// same launch also carries ncols CTAs that each own a strip of colw columns
// and add g*x*rstd over every row of the strip in a fixed order, writing dw
// directly; the row chunks then only write dx, and no partial rows, workspace
// or second kernel are used.  The order of the dw sum depends on T, H and the
// layout only, so dw no longer depends on the SM count.
#pragma once

#include <atomic>

#include "launch.h"

namespace crmsn {

#ifdef CRMSN_DEBUG
constexpr unsigned DBG_ASYNC_COPY_KIND = DBG_ASYNC_COPY;
#else
constexpr unsigned DBG_ASYNC_COPY_KIND = 0;
#endif

// Per-thread asynchronous global -> shared copies.
__device__ __forceinline__ void cp_async_16(void *smem, const void *gmem)
{
    if (!dbg_shared(smem, 16) || !dbg_global(gmem, 16, false, DBG_ASYNC_COPY_KIND)) return;
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_4(void *smem, const void *gmem)
{
    if (!dbg_shared(smem, 4) || !dbg_global(gmem, 4, false, DBG_ASYNC_COPY_KIND)) return;
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Rows summed plainly per column before each compensated fold.
constexpr int kDwBlock = 16;

// VEC BF16 values from a 16-byte (4-byte) aligned shared-memory slot in one
// access.
template <int VEC>
__device__ __forceinline__ BVec<VEC> ld_smem_vec(const unsigned char *p)
{
    BVec<VEC> v;
    if (!dbg_shared(p, VEC * 2)) {
        for (int i = 0; i < VEC / 2; ++i) v.w[i] = 0u;
        return v;
    }
    if constexpr (VEC == 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        v.w[0] = u.x; v.w[1] = u.y; v.w[2] = u.z; v.w[3] = u.w;
    } else {
        v.w[0] = *reinterpret_cast<const uint32_t *>(p);
    }
    return v;
}

// One FP32 value, and one (sum, compensation) pair, in shared memory.
__device__ __forceinline__ void st_smem_f32(float *p, float v)
{
    if (dbg_shared(p, 4)) *p = v;
}
__device__ __forceinline__ void st_smem_pair(float *p, float h, float l)
{
    if (dbg_shared(p, 8)) *reinterpret_cast<float2 *>(p) = make_float2(h, l);
}
__device__ __forceinline__ float2 ld_smem_pair(const float *p)
{
    if (!dbg_shared(p, 8)) return make_float2(0.f, 0.f);
    return *reinterpret_cast<const float2 *>(p);
}

// Bytes of one ring stage: NT tensors x VPT vectors per thread.
__host__ __device__ constexpr int bwd_stage_bytes(int nt, int vpt, int vec, int threads)
{
    return nt * vpt * threads * vec * 2;
}

// VEC BF16 values through L2 only (the row chunks of the same launch may
// read them again).
template <int VEC>
__device__ __forceinline__ BVec<VEC> ld_l2(const uint16_t *p)
{
    BVec<VEC> v;
    if (!dbg_global(p, VEC * 2, false)) {
        for (int i = 0; i < VEC / 2; ++i) v.w[i] = 0u;
        return v;
    }
    if constexpr (VEC == 8)
        asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    else
        asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    return v;
}

// Rows in flight per thread in the column form.
constexpr int kColUnroll = 8;

// Column form: dw of strip `strip` (columns [strip*colw, strip*colw + colw)
// clipped to H) over all T rows.  A row's strip is read by colw/VEC
// consecutive lanes (one vector each), so a warp covers 32*VEC/colw rows per
// access and the CTA `slots` rows; row slot k takes rows k, k + slots, ...
// in order.  Each lane adds its rows' terms (g*x)*rstd -- g*x exact from the
// mixed-precision FMA -- into plain FP32 block sums folded into compensated
// pairs every kDwBlock rows, as the row chunks do.  The slots of a warp are
// then added in a butterfly (slot order fixed by the lane bits), and the
// warps' pairs in warp order by one thread per column.  Every step depends on
// T, H, colw and the block size only.  `scratch` holds warps x colw pairs.
template <int VEC>
__device__ void dw_columns(const BwdParams &p, int strip, float2 *scratch)
{
    constexpr int NW = VEC / 2;
    const int lpr = p.colw / VEC;                 // lanes per row strip (power of two <= 32)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int slots = nwarps * (32 / lpr);
    const int slot = warp * (32 / lpr) + lane / lpr;
    const int64_t col = (int64_t)strip * p.colw + (int64_t)(lane & (lpr - 1)) * VEC;
    const bool live = col < p.H;

    float acc[VEC], cmp[VEC];
    F2 blk[NW];
#pragma unroll
    for (int i = 0; i < VEC; ++i) { acc[i] = 0.f; cmp[i] = 0.f; }
#pragma unroll
    for (int i = 0; i < NW; ++i) blk[i] = f2(0.f);
    auto fold = [&]() {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float b = (i & 1) ? f2_hi(blk[i >> 1]) : f2_lo(blk[i >> 1]);
            float s2, err;
            two_sum(acc[i], b, s2, err);
            acc[i] = s2;
            cmp[i] = __fadd_rn(cmp[i], err);
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) blk[i] = f2(0.f);
    };

    if (live) {
        const uint16_t *gp = p.g + (int64_t)slot * p.ldg + col;
        const uint16_t *xp = p.x + (int64_t)slot * p.ldx + col;
        const int64_t gstep = (int64_t)slots * p.ldg, xstep = (int64_t)slots * p.ldx;
        int n = 0;                                // rows added since the last fold
        for (int64_t t = slot; t < p.T; t += (int64_t)kColUnroll * slots) {
            BVec<VEC> gv[kColUnroll], xv[kColUnroll];
            float rs[kColUnroll];
#pragma unroll
            for (int u = 0; u < kColUnroll; ++u) {
                if (t + (int64_t)u * slots < p.T) {
                    gv[u] = ld_l2<VEC>(gp + u * gstep);
                    xv[u] = ld_l2<VEC>(xp + u * xstep);
                    rs[u] = ld_f32_ro(p.rstd + t + (int64_t)u * slots);
                }
            }
#pragma unroll
            for (int u = 0; u < kColUnroll; ++u) {
                if (t + (int64_t)u * slots < p.T) {
                    const F2 rs2 = f2(rs[u]);
#pragma unroll
                    for (int e = 0; e < NW; ++e)
                        blk[e] = f2_fma(mul_bf16x2(gv[u].w[e], xv[u].w[e]), rs2, blk[e]);
                    if (++n == kDwBlock) { fold(); n = 0; }
                }
            }
            gp += kColUnroll * gstep;
            xp += kColUnroll * xstep;
        }
    }
    fold();

    // Slots of the warp: partners differ in one slot bit and add each
    // other's pairs (pair_add is symmetric, so both hold the same bits).
    for (int o = lpr; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float bh = __shfl_xor_sync(0xffffffffu, acc[i], o);
            const float bl = __shfl_xor_sync(0xffffffffu, cmp[i], o);
            pair_add(acc[i], cmp[i], bh, bl);
        }
    if (lane < lpr)
#pragma unroll
        for (int i = 0; i < VEC; ++i)
            st_smem_pair(reinterpret_cast<float *>(scratch + warp * p.colw + lane * VEC + i), acc[i], cmp[i]);
    __syncthreads();
    for (int c = threadIdx.x; c < p.colw; c += blockDim.x) {
        const int64_t j = (int64_t)strip * p.colw + c;
        if (j >= p.H) continue;
        const float2 s0 = ld_smem_pair(reinterpret_cast<const float *>(scratch + c));
        float h = s0.x, l = s0.y;
        for (int w = 1; w < nwarps; ++w) {
            const float2 sw = ld_smem_pair(reinterpret_cast<const float *>(scratch + w * p.colw + c));
            pair_add(h, l, sw.x, sw.y);
        }
        st_f32(p.dw + j, __fadd_rn(h, l));
    }
}

// WB: a BF16 weight kept as BF16 in shared memory (the bias added as each
// vector is read) instead of as the FP32 effective weight: half the bytes,
// which leaves room for a deeper ring on the widest rows (chosen per launch).
template <bool W32, bool GRES, int VEC, int VPT, bool SUB, int D, bool WB>
__global__ void __launch_bounds__(kBwdMaxThreads, 1)
k_rmsnorm_bwd(const BwdParams p)
{
    static_assert(!WB || (!W32 && VEC == 8), "a BF16 weight in shared memory needs 16-byte vectors");
    constexpr int NW = VEC / 2;
    constexpr int NT = GRES ? 3 : 2;
    constexpr int S = D + 1;                  // ring stages
    constexpr int VB = VEC * 2;               // bytes per vector
    // Multi-warp groups with a ring run the software-pipelined loop.
    constexpr bool PIPE = !SUB && D >= 1;
    __shared__ float red_h[PIPE ? 1 : kBwdMaxThreads], red_l[PIPE ? 1 : kBwdMaxThreads];
    __shared__ float tot_h[32], tot_l[32];
    // Per-warp row sums of the pipelined path: [row parity][group][warp].
    __shared__ __align__(16) float wsum[PIPE ? 2 * kBwdMaxGroups * kBwdMaxGroupWarps : 4];
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    // Programmatic dependent launch: wait for the preceding grid (and its
    // memory) before any global access; let the reduce grid be scheduled now
    // (it waits for this whole grid the same way).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    CRMSN_DEBUG_ENTER(p.dbg);

    // Column form: the first ncols CTAs each reduce one strip of dw.
    if ((int)blockIdx.x < p.ncols) {
        dw_columns<VEC>(p, blockIdx.x, reinterpret_cast<float2 *>(dyn_smem));
        return;
    }
    const int chunk = blockIdx.x - p.ncols;

    const int nthr = blockDim.x;
    const int tpr = p.tpr;
    const int rpc = p.rpc;
    const int grp = row_group(tpr, p.rpc);
    const int lane = threadIdx.x - grp * tpr;
    const int nvec = p.H / VEC;
    const int64_t r0 = (int64_t)chunk * p.T / p.nchunk;
    const int64_t r1 = (int64_t)(chunk + 1) * p.T / p.nchunk;
    const int64_t iters = (r1 - r0 + rpc - 1) / rpc;

    // Shared memory: ring [S][stage], then w_eff [VPT*tpr*VEC] (zero past H),
    // then the row-group combine area [rpc][H][2] (when rpc > 1).  w_eff is stored in two
    // planes of four values per vector (one plane for VEC == 2), so that the
    // 16-byte loads of a warp touch consecutive addresses; with WB the BF16
    // weight instead, one 16-byte vector per column vector.
    const int stage_bytes = bwd_stage_bytes(NT, VPT, VEC, nthr);
    unsigned char *ring = dyn_smem;
    float *wsm = reinterpret_cast<float *>(dyn_smem + (size_t)S * stage_bytes);
    float *comb = wsm + (WB ? VPT * tpr * VEC / 2 : VPT * tpr * VEC);
    uint16_t *const wsb = reinterpret_cast<uint16_t *>(wsm);
    const int wplane = VPT * tpr * 4;

    // This thread's slot of vector k of a tensor in a stage; the per-thread
    // base and the strides are computed once.
    unsigned char *const my_slot = ring + (size_t)threadIdx.x * VB;
    const int kstride = nthr * VB;
    auto slot = [&](int stage, int tensor, int k) -> unsigned char * {
        return my_slot + (size_t)stage * stage_bytes + (tensor * VPT + k) * kstride;
    };
    auto w_at = [&](int v, int i) -> float * {
        if constexpr (VEC == 8) return wsm + (i < 4 ? 0 : wplane) + v * 4 + (i & 3);
        else return wsm + v * VEC + i;
    };
    auto ld_w = [&](int k, F2 (&we)[NW]) {
        const int v = k * tpr + lane;
        if constexpr (WB) {
            if (!dbg_shared(wsb + v * VEC, 16)) {
                for (int e = 0; e < NW; ++e) we[e] = f2(0.f);
                return;
            }
            const uint4 a = *reinterpret_cast<const uint4 *>(wsb + v * VEC);
            we[0] = f2_bf16(a.x); we[1] = f2_bf16(a.y); we[2] = f2_bf16(a.z); we[3] = f2_bf16(a.w);
            if (p.bias != 0.f) {
#pragma unroll
                for (int e = 0; e < NW; ++e) we[e] = f2_add(we[e], f2(p.bias));
            }
            return;
        }
        if (VEC == 8 ? !dbg_shared(wsm + v * 4, 16) || !dbg_shared(wsm + wplane + v * 4, 16)
                     : !dbg_shared(wsm + v * VEC, 8)) {
            for (int e = 0; e < NW; ++e) we[e] = f2(0.f);
            return;
        }
        if constexpr (VEC == 8) {
            const float4 a = *reinterpret_cast<const float4 *>(wsm + v * 4);
            const float4 b = *reinterpret_cast<const float4 *>(wsm + wplane + v * 4);
            we[0] = f2(a.x, a.y); we[1] = f2(a.z, a.w); we[2] = f2(b.x, b.y); we[3] = f2(b.z, b.w);
        } else {
            const float2 a = *reinterpret_cast<const float2 *>(wsm + v * VEC);
            we[0] = f2(a.x, a.y);
        }
    };
    // Copies of the iterations in order: issue_next() issues iteration
    // `iss` (row r0 + grp + iss*rpc) into stage iss % S and advances; the
    // source pointers of this thread's first vector move by a row step.
    int64_t iss = 0, t_iss = r0 + grp;
    const uint16_t *g_iss = p.g + t_iss * p.ldg + (int64_t)lane * VEC;
    const uint16_t *x_iss = p.x + t_iss * p.ldx + (int64_t)lane * VEC;
    const uint16_t *r_iss = GRES ? p.gres + t_iss * p.ldgr + (int64_t)lane * VEC : nullptr;
    int st_iss = 0;
    auto issue_next = [&]() {
        if (t_iss < r1) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (k * tpr + lane < nvec) {
                    const int c = k * tpr * VEC;
                    if constexpr (VEC == 8) {
                        cp_async_16(slot(st_iss, 0, k), g_iss + c);
                        cp_async_16(slot(st_iss, 1, k), x_iss + c);
                        if constexpr (GRES) cp_async_16(slot(st_iss, 2, k), r_iss + c);
                    } else {
                        cp_async_4(slot(st_iss, 0, k), g_iss + c);
                        cp_async_4(slot(st_iss, 1, k), x_iss + c);
                        if constexpr (GRES) cp_async_4(slot(st_iss, 2, k), r_iss + c);
                    }
                }
            }
        }
        cp_async_commit();   // one group per iteration, empty or not
        ++iss;
        t_iss += rpc;
        g_iss += (int64_t)rpc * p.ldg;
        x_iss += (int64_t)rpc * p.ldx;
        if constexpr (GRES) r_iss += (int64_t)rpc * p.ldgr;
        st_iss = st_iss + 1 == S ? 0 : st_iss + 1;
    };

    // Prologue: the first D rows go in flight while the weight is prepared.
#pragma unroll
    for (int i = 0; i < D; ++i) issue_next();

    // Effective weight f32(w + bias) of this thread's columns, in shared
    // memory; group 0 writes it, the other groups read it after a barrier.
    // Columns past H (the last vectors of a row that does not fill the
    // layout) get a zero weight and zero ring slots, which the copies never
    // touch, so every shared-memory load below is unconditional and those
    // columns add exact zeros to m and dw.
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * tpr + lane;
        const int64_t c = (int64_t)v * VEC;
        if (v >= nvec) {
#pragma unroll
            for (int st = 0; st < S; ++st)
#pragma unroll
                for (int ti = 0; ti < NT; ++ti) {
                    if (!dbg_shared(slot(st, ti, k), VB)) continue;
                    if constexpr (VEC == 8)
                        *reinterpret_cast<uint4 *>(slot(st, ti, k)) = make_uint4(0u, 0u, 0u, 0u);
                    else
                        *reinterpret_cast<uint32_t *>(slot(st, ti, k)) = 0u;
                }
            if (grp == 0) {
                if constexpr (WB) {
                    if (dbg_shared(wsb + v * VEC, 16))
                        *reinterpret_cast<uint4 *>(wsb + v * VEC) = make_uint4(0u, 0u, 0u, 0u);
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) st_smem_f32(w_at(v, i), 0.f);
                }
            }
        } else if (grp == 0) {
            if constexpr (WB) {
                // The BF16 weight as it is; with a bias of +0 a -0 is stored as
                // +0, the value f32(w) + 0 of the FP32 form (a nonzero bias is
                // added at each read, with the same rounding; adding -0
                // changes nothing).
                const BVec<VEC> wb = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
                const bool plus_zero = __float_as_uint(p.bias) == 0u;
                uint32_t q[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    q[i] = wb.w[i];
                    if (plus_zero) {
                        if ((q[i] & 0xffffu) == 0x8000u) q[i] &= 0xffff0000u;
                        if ((q[i] >> 16) == 0x8000u) q[i] &= 0x0000ffffu;
                    }
                }
                if (dbg_shared(wsb + v * VEC, 16))
                    *reinterpret_cast<uint4 *>(wsb + v * VEC) = make_uint4(q[0], q[1], q[2], q[3]);
            } else if constexpr (W32) {
                float f[VEC];
                ld_f32_keep<VEC>(static_cast<const float *>(p.w) + c, f);
#pragma unroll
                for (int i = 0; i < VEC; ++i) st_smem_f32(w_at(v, i), __fadd_rn(f[i], p.bias));
            } else {
                BVec<VEC> wb = ld_keep<VEC>(static_cast<const uint16_t *>(p.w) + c);
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    st_smem_f32(w_at(v, 2 * i), __fadd_rn(bf_lo(wb.w[i]), p.bias));
                    st_smem_f32(w_at(v, 2 * i + 1), __fadd_rn(bf_hi(wb.w[i]), p.bias));
                }
            }
        }
    }
    if (rpc > 1) __syncthreads();

    // rstd of the group's rows, BL rows at a time: lane j of each block holds
    // the rstd of the block's j-th row (one load per lane, issued a whole
    // block ahead) and the row's value is broadcast with a shuffle.  BL is
    // the group width within a warp (tpr, a power of two, for sub-warp
    // groups; 32 otherwise).  rs_cur holds the block of the current
    // iteration, rs_nxt the next block.
    const int BL = tpr < 32 ? tpr : 32;
    const int bl = lane & (BL - 1);
    auto rs_block = [&](int64_t it0) -> float {
        const int64_t t = r0 + grp + (it0 + bl) * rpc;
        return t < r1 ? ld_f32_ro(p.rstd + t) : 0.f;
    };
    float rs_cur = rs_block(0), rs_nxt = rs_block(BL);
    // rstd of iteration i, i in the current (it's) or the next block; called
    // by every lane of the warp together.
    auto rs_of = [&](int64_t i, int64_t it) -> float {
        const float src = ((i ^ it) & ~(int64_t)(BL - 1)) == 0 ? rs_cur : rs_nxt;
        return __shfl_sync(0xffffffffu, src, (int)(i & (BL - 1)), BL);
    };
    auto rs_advance = [&](int64_t it) {
        if (((it + 1) & (BL - 1)) == 0) {
            rs_cur = rs_nxt;
            rs_nxt = rs_block(it + 1 + BL);
        }
    };

    float acc[VPT][VEC], cmp[VPT][VEC];
    F2 blk[VPT][NW];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) { acc[k][i] = 0.f; cmp[k][i] = 0.f; }
#pragma unroll
        for (int i = 0; i < NW; ++i) blk[k][i] = f2(0.f);
    }
    auto fold = [&]() {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                const float b = (i & 1) ? f2_hi(blk[k][i >> 1]) : f2_lo(blk[k][i >> 1]);
                float s2, err;
                two_sum(acc[k][i], b, s2, err);
                acc[k][i] = s2;
                cmp[k][i] = __fadd_rn(cmp[k][i], err);
            }
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int i = 0; i < NW; ++i) blk[k][i] = f2(0.f);
    };

    // Vector k of a row: dot2 += g*w*x (two FP32 lanes).
    auto dot_vec = [&](int stage, int k, const F2 (&we)[NW], F2 &dot2) {
        const BVec<VEC> gv = ld_smem_vec<VEC>(slot(stage, 0, k));
        const BVec<VEC> xv = ld_smem_vec<VEC>(slot(stage, 1, k));
#pragma unroll
        for (int e = 0; e < NW; ++e)
            dot2 = f2_fma(f2_mul(f2_bf16(gv.w[e]), we[e]), f2_bf16(xv.w[e]), dot2);
    };
    // Vector k of a row with rstd rs2: dot2 += (g*x)*w, and the dw terms
    // (g*x)*rstd into the block sums, from the exact products g*x.
    auto dot_dw_vec = [&](int stage, int k, const F2 (&we)[NW], F2 rs2, F2 &dot2) {
        const BVec<VEC> gv = ld_smem_vec<VEC>(slot(stage, 0, k));
        const BVec<VEC> xv = ld_smem_vec<VEC>(slot(stage, 1, k));
#pragma unroll
        for (int e = 0; e < NW; ++e) {
            const F2 gx = mul_bf16x2(gv.w[e], xv.w[e]);
            dot2 = f2_fma(gx, we[e], dot2);
            blk[k][e] = f2_fma(gx, rs2, blk[k][e]);
        }
    };
    // Vector k of row t: dx = rstd*(g*w) - x*(rstd^3*m) (+ g_residual), and
    // with with_dw the dw terms g*x*rstd (g*x is exact in FP32) into the block
    // sums.
    auto dx_vec = [&](bool with_dw, uint16_t *dxrow, int stage, int k, const F2 (&we)[NW], F2 rs2, F2 nc3) {
        const int v = k * tpr + lane;
        const BVec<VEC> gv = ld_smem_vec<VEC>(slot(stage, 0, k));
        const BVec<VEC> xv = ld_smem_vec<VEC>(slot(stage, 1, k));
        BVec<VEC> rv;
        if constexpr (GRES) rv = ld_smem_vec<VEC>(slot(stage, 2, k));
        BVec<VEC> o;
#pragma unroll
        for (int e = 0; e < NW; ++e) {
            const F2 g2 = f2_bf16(gv.w[e]);
            const F2 x2 = f2_bf16(xv.w[e]);
            F2 d2 = f2_fma(x2, nc3, f2_mul(rs2, f2_mul(g2, we[e])));
            if constexpr (GRES) d2 = f2_add(d2, f2_bf16(rv.w[e]));
            o.w[e] = bf16_f2(d2);
            if (with_dw) blk[k][e] = f2_fma(f2_mul(g2, x2), rs2, blk[k][e]);
        }
        if (v < nvec) st_stream<VEC>(dxrow + k * tpr * VEC, o);
    };
    // rstd*1 and -rstd^3*m for a row with rstd rs and sum of g*w*x `sum`.
    // m = sum / H as sum * RN(1/H): exact for a power-of-two H, within one
    // FP32 ulp otherwise (m only scales dx's small second term).
    const float inv_h = __frcp_rn((float)p.H);
    auto coefs = [&](float rs, float sum, F2 &rs2, F2 &nc3) {
        const float m = __fmul_rn(sum, inv_h);
        rs2 = f2(rs);
        nc3 = f2(-__fmul_rn(__fmul_rn(__fmul_rn(rs, rs), rs), m));
    };

    if constexpr (PIPE) {
        // Multi-warp groups, software-pipelined.  Iteration `it` forms row
        // it+1's sum of g*w*x and adds it up inside each warp (butterfly:
        // every lane ends with the same bits) while it writes row it's dx,
        // reading each weight vector once for both rows; one CTA barrier per
        // row publishes the per-warp sums, and every thread then adds its
        // group's warp sums itself in a fixed pairwise order.  Plain FP32
        // sums (m only scales the small second term of dx).  The ring holds
        // rows it and it+1 plus D - 1 rows ahead.
        const int wg = lane >> 5;
        for (int i = threadIdx.x; i < 2 * kBwdMaxGroups * kBwdMaxGroupWarps; i += nthr)
            if (i % kBwdMaxGroupWarps >= (tpr >> 5)) wsum[i] = 0.f;   // never-written warp slots
        auto publish = [&](int64_t i, F2 d2) {
            float sum = __fadd_rn(f2_lo(d2), f2_hi(d2));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
            if ((lane & 31) == 0) wsum[((int)(i & 1) * kBwdMaxGroups + grp) * kBwdMaxGroupWarps + wg] = sum;
        };
        // Sum of the group's warp slots in a fixed pairwise tree over 8 slots
        // (groups of at most 8 warps) or 16; the unused slots hold zeros.
        const bool narrow_group = tpr <= 256;
        auto group_total = [&](int64_t i) -> float {
            const float4 *q = reinterpret_cast<const float4 *>(
                wsum + ((int)(i & 1) * kBwdMaxGroups + grp) * kBwdMaxGroupWarps);
            float v[kBwdMaxGroupWarps];
            if (narrow_group) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float4 f = q[j];
                    v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
                }
#pragma unroll
                for (int w = 1; w < 8; w <<= 1)
#pragma unroll
                    for (int j = 0; j + w < 8; j += 2 * w) v[j] = __fadd_rn(v[j], v[j + w]);
                return v[0];
            }
#pragma unroll
            for (int j = 0; j < kBwdMaxGroupWarps / 4; ++j) {
                const float4 f = q[j];
                v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
            }
#pragma unroll
            for (int w = 1; w < kBwdMaxGroupWarps; w <<= 1)
#pragma unroll
                for (int j = 0; j + w < kBwdMaxGroupWarps; j += 2 * w) v[j] = __fadd_rn(v[j], v[j + w]);
            return v[0];
        };

        // The dw terms of a row are taken in its sum phase, from the exact
        // products g*x; block sums fold after every kDwBlock rows.
        cp_async_wait<D - 1>();              // row 0 landed
        {
            const F2 rs2 = f2(rs_of(0, 0));
            F2 dot2 = f2(0.f);
            if (r0 + grp < r1) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    F2 we[NW];
                    ld_w(k, we);
                    dot_dw_vec(0, k, we, rs2, dot2);
                }
            }
            publish(0, dot2);
        }
        __syncthreads();
        float tot = group_total(0);
        int64_t t = r0 + grp;                // row of iteration it
        uint16_t *dxrow = p.dx + t * p.lddx + (int64_t)lane * VEC;
        int st = 0;                          // its stage
        // One iteration; `checked` = false when rows it and it+1 are known to
        // be live (every iteration but the last two), so the body has no
        // liveness tests.
        auto step = [&](int64_t it, bool checked) {
            issue_next();                    // iteration it + D
            cp_async_wait<D - 1>();          // this thread's copies of rows it, it+1 landed
            const float rs = rs_of(it, it);
            const F2 rsn2 = f2(rs_of(it + 1, it));
            const bool live = !checked || t < r1;
            const bool live_n = !checked || t + rpc < r1;
            const int st_n = st + 1 == S ? 0 : st + 1;
            F2 rs2, nc3;
            coefs(rs, tot, rs2, nc3);
            F2 dot2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                F2 we[NW];
                ld_w(k, we);
                if (live_n) dot_dw_vec(st_n, k, we, rsn2, dot2);
                if (live) dx_vec(false, dxrow, st, k, we, rs2, nc3);
            }
            publish(it + 1, dot2);
            rs_advance(it);
            t += rpc;
            dxrow += (int64_t)rpc * p.lddx;
            st = st_n;
            __syncthreads();
            tot = group_total(it + 1);
        };
        // Steps in blocks that end where the block sums fold (after the step
        // with (it + 2) % kDwBlock == 0), so the fold never sits inside the
        // per-row body; the last two steps check liveness.
        int64_t it = 0;
        const int64_t nfast = iters > 2 ? iters - 2 : 0;
        while (it < iters) {
            int64_t stop = it + (kDwBlock - (it + 2) % kDwBlock);
            if (stop > iters) stop = iters;
            const int64_t fstop = stop < nfast ? stop : nfast;
            for (; it < fstop; ++it) step(it, false);
            for (; it < stop; ++it) step(it, true);
            if ((it + 1) % kDwBlock == 0) fold();
        }
    } else {
        int64_t t = r0 + grp;                // row of iteration it
        uint16_t *dxrow = p.dx + t * p.lddx + (int64_t)lane * VEC;
        int st = 0;                          // its stage
        for (int64_t it = 0; it < iters; ++it) {
            issue_next();                    // iteration it + D: keep D rows ahead in flight
            cp_async_wait<D>();              // this thread's copies of row `it` landed
            const float rs = rs_of(it, it);
            const bool live = t < r1;
            F2 dot2 = f2(0.f);
            if (live) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    F2 we[NW];
                    ld_w(k, we);
                    dot_vec(st, k, we, dot2);
                }
            }
            float h, l;
            two_sum(f2_lo(dot2), f2_hi(dot2), h, l);
            if constexpr (SUB)
                pair_reduce_lanes(h, l, tpr);
            else
                group_sum_pair(h, l, red_h, red_l, tot_h, tot_l, grp, tpr);
            if (live) {
                F2 rs2, nc3;
                coefs(rs, __fadd_rn(h, l), rs2, nc3);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    F2 we[NW];
                    ld_w(k, we);
                    dx_vec(true, dxrow, st, k, we, rs2, nc3);
                }
            }
            if ((it + 1) % kDwBlock == 0) fold();
            rs_advance(it);
            t += rpc;
            dxrow += (int64_t)rpc * p.lddx;
            st = st + 1 == S ? 0 : st + 1;
        }
    }
    fold();
    cp_async_wait<0>();
    if (p.ncols > 0) return;                 // dw comes from the column CTAs

    // Combine the CTA's row groups in group order, then write the partial row.
    // With several groups, every group stores its (sum, compensation) pairs in
    // comb[group][column], and after one barrier each thread adds whole
    // columns over the groups in group order (the same order, so the same
    // bits, as one group adding the others in turn, but spread over the CTA).
    float *prow = p.part + (int64_t)chunk * p.H;
    if (rpc > 1) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            if (v < nvec)
#pragma unroll
                for (int i = 0; i < VEC; ++i)
                    st_smem_pair(comb + ((int64_t)grp * p.H + (int64_t)v * VEC + i) * 2, acc[k][i], cmp[k][i]);
        }
        __syncthreads();
        for (int col = threadIdx.x; col < p.H; col += nthr) {
            const float2 c0 = ld_smem_pair(comb + (int64_t)col * 2);
            float h = c0.x, l = c0.y;
            for (int gi = 1; gi < rpc; ++gi) {
                const float2 c = ld_smem_pair(comb + ((int64_t)gi * p.H + col) * 2);
                pair_add(h, l, c.x, c.y);
            }
            st_f32(prow + col, __fadd_rn(h, l));
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + lane;
            if (v < nvec)
#pragma unroll
                for (int i = 0; i < VEC; ++i)
                    st_f32(prow + (int64_t)v * VEC + i, __fadd_rn(acc[k][i], cmp[k][i]));
        }
    }
}

// Dynamic shared memory of one CTA for a layout and prefetch depth D.
inline size_t bwd_smem_bytes(bool wb, bool gres, int vec, int vpt, int threads, int rpc, int H, int D)
{
    return (size_t)(D + 1) * bwd_stage_bytes(gres ? 3 : 2, vpt, vec, threads) +
           (size_t)vpt * (threads / rpc) * vec * (wb ? 2 : 4) +
           (rpc > 1 ? (size_t)rpc * H * 2 * sizeof(float) : 0);
}

// The most shared memory a CTA may ask for, and the most the backward's
// CTAs on one SM are given together when a depth is chosen (measured: two
// CTAs taking 226 KB with g_residual at H = 4096 ran at 103.7 us, two of
// 89 KB at 94.7 us; 200 KB at H = 5120 was still the fastest).
constexpr size_t kBwdSmemMax = 227 * 1024;
constexpr size_t kBwdSmemPerSm = 208 * 1024;

// One instantiation: its residency (CTAs per SM for a block size and
// shared-memory size, computed once per key and remembered) and its launch
// with a chunk count of at most per_sm x SMs (and at most one chunk per row
// group).
template <bool W32, bool GRES, int VEC, int VPT, bool SUB, int D, bool WB>
struct BwdInst {
    static constexpr auto kern = k_rmsnorm_bwd<W32, GRES, VEC, VPT, SUB, D, WB>;

    static cudaError_t occupancy(const BwdParams &p, int *per_sm)
    {
        const int threads = p.tpr * p.rpc;
        const size_t smem = bwd_smem_bytes(WB, GRES, VEC, VPT, threads, p.rpc, p.H, D);
        static std::atomic<int> opted[kOptInDevices];
        cudaError_t e = opt_in_smem(kern, smem, opted);
        if (e != cudaSuccess) return e;
        // threads << 40 | shared-memory bytes << 8 | CTAs per SM
        static std::atomic<long long> cached{0};
        const long long key = ((long long)threads << 40) | ((long long)smem << 8);
        const long long c = cached.load(std::memory_order_relaxed);
        if ((c & ~0xffLL) == key && (c & 0xff) > 0) {
            *per_sm = (int)(c & 0xff);
            return cudaSuccess;
        }
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem);
        if (e != cudaSuccess) return e;
        if (n > 255) n = 255;
        if (n > 0) cached.store(key | n, std::memory_order_relaxed);
        *per_sm = n;
        return cudaSuccess;
    }

    // Row chunks: as many as resident CTAs (per_sm x SMs) less the strip
    // CTAs, but at least a third of the resident CTAs, and at most one chunk
    // per row group.  Strip and chunk CTAs run side by side: a strip CTA
    // reads 4 bytes per row and column of its strip, a chunk CTA 6 (8 with
    // g_residual) per row and column of its rows.
    static cudaError_t launch(BwdParams p, int per_sm, int sms, int *nchunk_out, cudaStream_t s)
    {
        const int threads = p.tpr * p.rpc;
        size_t smem = bwd_smem_bytes(WB, GRES, VEC, VPT, threads, p.rpc, p.H, D);
        const size_t col_smem = (size_t)(threads / 32) * p.colw * sizeof(float2);
        if (p.ncols > 0 && col_smem > smem) smem = col_smem;
        const int64_t by_rows = (p.T + p.rpc - 1) / p.rpc;
        const int64_t resident = (int64_t)per_sm * sms;
        int64_t cap = resident - p.ncols;
        if (cap < (resident + 2) / 3) cap = (resident + 2) / 3;
        p.nchunk = (int)(by_rows < cap ? by_rows : cap);
        *nchunk_out = p.nchunk;
        return launch_pdl(kern, dim3((unsigned)(p.ncols + p.nchunk)), dim3(threads), smem, s, p);
    }
};

// Calls f(BwdInst<...>{}) for the instantiation of a layout (SUB groups with
// VPT 1|2; multi-warp groups with VPT 1|2|4 for 16-byte vectors, 1|2|4|8|16
// for 4-byte vectors; the unpipelined D = 0 form only for 32 elements per
// thread; the BF16 weight in shared memory (wb) only for a BF16 weight with
// 32 elements per thread in 16-byte vectors and a ring).
template <bool W32, bool GRES, int VEC, int D, typename F>
cudaError_t with_bwd_inst(const Layout &L, bool wb, F &&f)
{
    constexpr int V32 = 32 / VEC;
    if constexpr (D == 0) {
        if (!wb && !L.sub && L.vpt == V32) return f(BwdInst<W32, GRES, VEC, V32, false, 0, false>{});
        return cudaErrorInvalidConfiguration;
    } else {
        if constexpr (!W32 && VEC == 8) {
            if (wb) {
                if (!L.sub && L.vpt == 4) return f(BwdInst<W32, GRES, VEC, 4, false, D, true>{});
                return cudaErrorInvalidConfiguration;
            }
        }
        if (wb) return cudaErrorInvalidConfiguration;
        if (L.sub) {
            if (L.vpt == 1) return f(BwdInst<W32, GRES, VEC, 1, true, D, false>{});
            if (L.vpt == 2) return f(BwdInst<W32, GRES, VEC, 2, true, D, false>{});
        } else {
            if (L.vpt == 1) return f(BwdInst<W32, GRES, VEC, 1, false, D, false>{});
            if (L.vpt == 2) return f(BwdInst<W32, GRES, VEC, 2, false, D, false>{});
            if (L.vpt == 4) return f(BwdInst<W32, GRES, VEC, 4, false, D, false>{});
            if constexpr (VEC == 2) {
                if (L.vpt == 8) return f(BwdInst<W32, GRES, VEC, 8, false, D, false>{});
                if (L.vpt == 16) return f(BwdInst<W32, GRES, VEC, 16, false, D, false>{});
            }
        }
        return cudaErrorInvalidConfiguration;
    }
}

template <bool W32, bool GRES, int VEC, typename F>
cudaError_t with_bwd_depth(int D, const Layout &L, bool wb, F &&f)
{
    switch (D) {
        case 3: return with_bwd_inst<W32, GRES, VEC, 3>(L, wb, f);
        case 2: return with_bwd_inst<W32, GRES, VEC, 2>(L, wb, f);
        case 1: return with_bwd_inst<W32, GRES, VEC, 1>(L, wb, f);
        default: return with_bwd_inst<W32, GRES, VEC, 0>(L, wb, f);
    }
}

// Prefetch depth and residency: among the depths whose ring fits a CTA's
// shared memory, the one with the most rows in flight per SM (CTAs per SM --
// capped at bwd_max_ctas_per_sm(H) and at what kBwdSmemPerSm holds --
// times the depth), the larger CTA count on a tie; D = 0 (no ring) only
// when no ring fits.  The pipelined loop overlaps the loads with the
// arithmetic only from D = 2 on (it waits for row i + 1 while row i + D is
// issued); where the FP32 weight leaves it at D <= 1 (a BF16 weight, 32
// elements per thread: H above about 14500, or with g_residual above about
// 10500) the weight is held as BF16 if that gives a deeper ring (measured
// at T = H = 16384: 310 -> 271 us, with g_residual 459 -> 363 us; where
// the depth is the same it costs about 5 %, the conversion at each read).
template <bool W32, bool GRES, int VEC>
cudaError_t launch_bwd_vec(const BwdParams &p, const Layout &L, int sms, int *nc, cudaStream_t s)
{
    const int threads = p.tpr * p.rpc;
    const int cap = bwd_max_ctas_per_sm(p.H);
    auto choose = [&](bool wb, int &best_d, int &best_n) -> cudaError_t {
        best_d = -1;
        best_n = 1;
        long best_score = -1;
        for (int d = 3; d >= 1; --d) {
            const size_t smem = bwd_smem_bytes(wb, GRES, VEC, L.vpt, threads, p.rpc, p.H, d);
            if (smem > kBwdSmemMax) continue;
            int n = 0;
            cudaError_t e = with_bwd_depth<W32, GRES, VEC>(d, L, wb, [&](auto inst) {
                return decltype(inst)::occupancy(p, &n);
            });
            if (e != cudaSuccess) return e;
            if (n > cap) n = cap;
            const int by_budget = (int)(kBwdSmemPerSm / (smem + 1024));
            if (n > by_budget) n = by_budget > 0 ? by_budget : 1;
            if (n < 1) continue;
            const long score = (long)n * d * 16 + n;
            if (score > best_score) {
                best_score = score;
                best_d = d;
                best_n = n;
            }
        }
        return cudaSuccess;
    };
    int best_d = -1, best_n = 1;
    bool wb = false;
    cudaError_t e = choose(false, best_d, best_n);
    if (e != cudaSuccess) return e;
    if (!W32 && VEC == 8 && !L.sub && L.vpt == 4 && best_d <= 1) {
        int d2 = -1, n2 = 1;
        e = choose(true, d2, n2);
        if (e != cudaSuccess) return e;
        if (d2 > best_d) {
            wb = true;
            best_d = d2;
            best_n = n2;
        }
    }
    if (best_d < 0) {
        best_d = 0;
        e = with_bwd_depth<W32, GRES, VEC>(0, L, false, [&](auto inst) {
            return decltype(inst)::occupancy(p, &best_n);
        });
        if (e != cudaSuccess) return e;
        if (best_n < 1) return cudaErrorInvalidConfiguration;
        if (best_n > cap) best_n = cap;
    }
    return with_bwd_depth<W32, GRES, VEC>(best_d, L, wb, [&](auto inst) {
        return decltype(inst)::launch(p, best_n, sms, nc, s);
    });
}

template <bool W32, bool GRES>
cudaError_t launch_bwd_weight(const BwdParams &p, const Layout &L, int sms, int *nc, cudaStream_t s)
{
    if (L.vec == 8) return launch_bwd_vec<W32, GRES, 8>(p, L, sms, nc, s);
    if (L.vec == 2) return launch_bwd_vec<W32, GRES, 2>(p, L, sms, nc, s);
    return cudaErrorInvalidConfiguration;
}

}  // namespace crmsn
