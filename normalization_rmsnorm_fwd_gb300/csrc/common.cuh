// common.cuh -- device helpers shared by the RMSNorm kernels (sm_103a).
//
// BF16 vectors are held as packed 32-bit words (two BF16 per word, element
// 2i in the low half).  Streaming tensors are read and written with the
// evict-first cache hint; weights and broadcast style rows go through the
// read-only path.  All conversions round to nearest even with one PTX
// instruction; FP32 arithmetic is IEEE (the library is built without fast
// math).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace crmsn {

// ------------------------------------------------------ debug bounds guard --
// A build with -DCRMSN_DEBUG checks every global load and store of the
// kernels against the byte ranges of the call's tensors (all of them
// readable; outputs and the workspace writable) and every access to dynamic
// shared memory against the size the launch gave.  An access outside them is
// skipped (a load gives zeros) and the first one is recorded in a device word
// that crmsn_debug_status() reads back; nothing traps.  In the normal build
// every check is the constant true and the range table is not passed.
constexpr int kDebugMaxRanges = 12;
struct DebugRanges {
    unsigned long long *word;                    // first violation (0: none)
    unsigned long long lo[kDebugMaxRanges], hi[kDebugMaxRanges];
    unsigned writable;                           // bit i: range i may be written
    int n;
};

#ifdef CRMSN_DEBUG
// Kinds of access in a violation word: bits 62..56 kind, 55..32 the CTA,
// 31..22 the thread, 21..0 the low bits of the global address (of the byte
// offset for shared memory); bit 63 set.
enum : unsigned { DBG_LOAD = 1, DBG_STORE = 2, DBG_ASYNC_COPY = 3, DBG_SMEM = 4 };
static __shared__ DebugRanges dbg_ranges;
extern __shared__ __align__(16) unsigned char dbg_dyn_smem[];

// Every kernel's first step: the call's ranges into shared memory.
__device__ __forceinline__ void dbg_enter(const DebugRanges &r)
{
    if (threadIdx.x == 0) dbg_ranges = r;
    __syncthreads();
}
static __device__ __noinline__ void dbg_record(unsigned kind, unsigned long long where)
{
    const unsigned long long w = (1ull << 63) | ((unsigned long long)kind << 56) |
                                 ((unsigned long long)(blockIdx.x & 0xffffffu) << 32) |
                                 ((unsigned long long)(threadIdx.x & 0x3ffu) << 22) |
                                 (where & 0x3fffffull);
    if (dbg_ranges.word) atomicCAS(dbg_ranges.word, 0ull, w);
}
__device__ __forceinline__ bool dbg_global(const void *p, int bytes, bool write, unsigned kind = 0)
{
    const unsigned long long a = (unsigned long long)p, e = a + (unsigned long long)bytes;
    for (int i = 0; i < dbg_ranges.n; ++i)
        if (a >= dbg_ranges.lo[i] && e <= dbg_ranges.hi[i] && (!write || ((dbg_ranges.writable >> i) & 1u)))
            return true;
    dbg_record(kind ? kind : (write ? DBG_STORE : DBG_LOAD), a);
    return false;
}
__device__ __forceinline__ bool dbg_shared(const void *p, int bytes)
{
    unsigned size;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
    const long long off = (long long)((const unsigned char *)p - dbg_dyn_smem);
    if (off >= 0 && off + bytes <= (long long)size) return true;
    dbg_record(DBG_SMEM, (unsigned long long)off);
    return false;
}
#define CRMSN_DEBUG_ENTER(r) ::crmsn::dbg_enter(r)
#else
__device__ __forceinline__ constexpr bool dbg_global(const void *, int, bool, unsigned = 0) { return true; }
__device__ __forceinline__ constexpr bool dbg_shared(const void *, int) { return true; }
#define CRMSN_DEBUG_ENTER(r) ((void)0)
#endif

// ------------------------------------------------------------ BF16 / FP8 --

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed BF16 pair (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two floats -> packed FP8 pair (lo in bits 0..7), round to nearest even,
// saturating to the largest finite value.  KIND 0 = E4M3FN, 1 = E5M2.
template <int KIND>
__device__ __forceinline__ uint32_t pack_fp8(float lo, float hi)
{
    uint16_t r;
    if constexpr (KIND == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------ packed FP32 pairs --
// Blackwell executes two FP32 operations per instruction on a register pair
// (add/mul/fma .rn.f32x2, reached through the float2 builtins, which leave
// the pairing of registers to the compiler); each lane rounds exactly like
// the scalar IEEE operation, subnormal operands and results included (no
// flush to zero), so these only halve the instruction count.

using F2 = float2;

__device__ __forceinline__ F2 f2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ F2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float f2_lo(F2 a) { return a.x; }
__device__ __forceinline__ float f2_hi(F2 a) { return a.y; }
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) { return __ffma2_rn(a, b, c); }
// Packed BF16 pair -> FP32 pair (exact).
__device__ __forceinline__ F2 f2_bf16(uint32_t w) { return f2(bf_lo(w), bf_hi(w)); }

// ------------------------------------------------- mixed-precision BF16 --
// Blackwell's mixed-precision FMA takes BF16 multiplicands straight from the
// halves of a packed word (FP32 addend and result), so products of BF16
// values need no unpacking.  A product of two BF16 values has at most 16
// significant bits, so it is exact in FP32.

// (lo(a)*lo(b), hi(a)*hi(b)) of two packed BF16 pairs, exact.
__device__ __forceinline__ F2 mul_bf16x2(uint32_t a, uint32_t b)
{
    float lo, hi;
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %4;\n\tfma.rn.f32.bf16 %1, a1, b1, %4;\n}"
        : "=f"(lo), "=f"(hi) : "r"(a), "r"(b), "f"(-0.f));
    return f2(lo, hi);
}

// (lo(h) + c, hi(h) + c): the FP32 sums of the halves of a packed BF16 pair
// and an FP32 value, one rounding each (the same bits as unpacking first).
__device__ __forceinline__ F2 add_bf16x2(uint32_t h, float c)
{
    float lo, hi;
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "add.rn.f32.bf16 %0, h0, %3;\n\tadd.rn.f32.bf16 %1, h1, %3;\n}"
        : "=f"(lo), "=f"(hi) : "r"(h), "f"(c));
    return f2(lo, hi);
}

// lo += lo(h), hi += hi(h) for a packed BF16 pair h (one rounding each).
__device__ __forceinline__ void acc_bf16x2(uint32_t h, float &lo, float &hi)
{
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "add.rn.f32.bf16 %0, h0, %0;\n\tadd.rn.f32.bf16 %1, h1, %1;\n}"
        : "+f"(lo), "+f"(hi) : "r"(h));
}

// lo += lo(h)^2, hi += hi(h)^2 for a packed BF16 pair h (each square exact,
// one rounding per addition).
__device__ __forceinline__ void sq_acc_bf16x2(uint32_t h, float &lo, float &hi)
{
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, h0, h0, %0;\n\tfma.rn.f32.bf16 %1, h1, h1, %1;\n}"
        : "+f"(lo), "+f"(hi) : "r"(h));
}

// ------------------------------------------------------ division by a scale --
// v / s rounded to nearest (the IEEE quotient) for a pair v and one divisor s
// whose reciprocal r = RN(1/s) is known, in five packed instructions:
// q = RN(v*r), then twice q = RN(q + (v - s*q)*r) with the remainder v - s*q
// formed exactly by a fused multiply-add.  Markstein's theorem (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): when r is the correctly rounded
// reciprocal and q is within one ulp of v/s, the remainder is exact and the
// corrected quotient is correctly rounded; the first correction brings
// RN(v*r) (within 1.5 ulps) within one ulp.  This needs the quotient and the
// remainder to be normal FP32 numbers: a remainder below 2^-126 is rounded
// to the subnormal grid, so dividends below 2^-96 (for |s| >= 2^-60) are
// left to the caller, whose FP8 codes are zero there.
__device__ __forceinline__ F2 f2_div_recip(F2 v, float s, float r)
{
    const F2 ns = f2(-s), r2 = f2(r);
    F2 q = f2_mul(v, r2);
    F2 e = f2_fma(q, ns, v);
    q = f2_fma(e, r2, q);
    e = f2_fma(q, ns, v);
    return f2_fma(e, r2, q);
}

// Division by one scale s (the 1x128 block quantiser's f32(amax / 448),
// whose codes must equal those of the IEEE quotient bit for bit).  For |s|
// in [2^-60, 2^60] the quotient is the IEEE quotient v / s whenever
// |v| >= 2^-96 and the quotient is finite; a smaller dividend has a quotient
// below 2^-36, which every FP8 format rounds to zero whatever its last bits,
// and a quotient beyond the FP32 range comes out as NaN instead of an
// infinity.  Other scales use the IEEE division itself.
struct DivScale {
    float s, r;
    bool fast;
    __device__ __forceinline__ explicit DivScale(float s_) : s(s_), r(0.f), fast(false)
    {
        const float a = fabsf(s_);
        fast = a >= 0x1p-60f && a <= 0x1p60f;
        if (fast) r = __frcp_rn(s_);
    }
    __device__ __forceinline__ void div(F2 v, float &lo, float &hi) const
    {
        if (fast) {
            const F2 q = f2_div_recip(v, s, r);
            lo = f2_lo(q);
            hi = f2_hi(q);
        } else {
            lo = __fdiv_rn(f2_lo(v), s);
            hi = __fdiv_rn(f2_hi(v), s);
        }
    }
};
// FP32 pair -> packed BF16 pair, round to nearest even.
__device__ __forceinline__ uint32_t bf16_f2(F2 a) { return pack_bf16(f2_lo(a), f2_hi(a)); }

// Row group of a thread when a CTA holds `rpc` groups of `tpr` threads: no
// division for one group per CTA or a power-of-two group width (every layout
// but a few narrow ones).
__device__ __forceinline__ int row_group(int tpr, int rpc)
{
    if (rpc == 1) return 0;
    if ((tpr & (tpr - 1)) == 0) return (int)threadIdx.x >> (31 - __clz(tpr));
    return (int)threadIdx.x / tpr;
}

// ------------------------------------------------------------ vectors ----
// VEC BF16 elements = VEC/2 packed words.  VEC is 8 (16-byte accesses) or 2
// (4-byte accesses).

template <int VEC>
struct BVec {
    uint32_t w[VEC / 2];
};

template <int VEC>
__device__ __forceinline__ BVec<VEC> ld_stream(const uint16_t *p)
{
    BVec<VEC> v;
    if (!dbg_global(p, VEC * 2, false)) {
        for (int i = 0; i < VEC / 2; ++i) v.w[i] = 0u;
        return v;
    }
    if constexpr (VEC == 8)
        asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    else
        asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    return v;
}

template <int VEC>
__device__ __forceinline__ BVec<VEC> ld_keep(const uint16_t *p)
{
    BVec<VEC> v;
    if (!dbg_global(p, VEC * 2, false)) {
        for (int i = 0; i < VEC / 2; ++i) v.w[i] = 0u;
        return v;
    }
    if constexpr (VEC == 8)
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    else
        asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    return v;
}

template <int VEC>
__device__ __forceinline__ void st_stream(uint16_t *p, const BVec<VEC> &v)
{
    if (!dbg_global(p, VEC * 2, true)) return;
    if constexpr (VEC == 8)
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                     :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                     : "memory");
    else
        asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v.w[0]) : "memory");
}

// VEC FP8 codes (VEC bytes) stored from VEC/4 (VEC=8) or a half word (VEC=2).
template <int VEC>
__device__ __forceinline__ void st_fp8(uint8_t *p, const uint32_t (&c)[VEC / 2])
{
    // c[i] holds the FP8 pair of elements 2i, 2i+1 in its low 16 bits.
    if (!dbg_global(p, VEC, true)) return;
    if constexpr (VEC == 8) {
        uint32_t a = (c[0] & 0xffffu) | (c[1] << 16);
        uint32_t b = (c[2] & 0xffffu) | (c[3] << 16);
        asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(a), "r"(b) : "memory");
    } else {
        uint16_t a = (uint16_t)c[0];
        asm volatile("st.global.cs.u16 [%0], %1;" :: "l"(p), "h"(a) : "memory");
    }
}

// VEC FP32 weights (read-only path).
template <int VEC>
__device__ __forceinline__ void ld_f32_keep(const float *p, float (&f)[VEC])
{
    if (!dbg_global(p, VEC * 4, false)) {
        for (int i = 0; i < VEC; ++i) f[i] = 0.f;
        return;
    }
    if constexpr (VEC == 8) {
        asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]) : "l"(p));
        asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7]) : "l"(p + 4));
    } else {
        asm volatile("ld.global.nc.v2.f32 {%0,%1}, [%2];" : "=f"(f[0]), "=f"(f[1]) : "l"(p));
    }
}

// One FP32 value through the read-only path, and one plain FP32 store.
__device__ __forceinline__ float ld_f32_ro(const float *p)
{
    if (!dbg_global(p, 4, false)) return 0.f;
    return __ldg(p);
}
__device__ __forceinline__ void st_f32(float *p, float v)
{
    if (!dbg_global(p, 4, true)) return;
    *p = v;
}

// ------------------------------------------------- compensated reductions --
// A value is carried as an unevaluated pair (hi, lo); TwoSum keeps the
// rounding error of every addition, so a tree of pair additions returns the
// sum with an error of a few units in the last place of lo.  TwoSum is
// symmetric in its operands, so both partners of a butterfly exchange end up
// with identical pairs.

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void pair_add(float &h, float &l, float bh, float bl)
{
    float s, e;
    two_sum(h, bh, s, e);
    e = __fadd_rn(e, __fadd_rn(l, bl));
    h = __fadd_rn(s, e);
    l = __fsub_rn(e, __fsub_rn(h, s));
}

// Butterfly over `width` lanes (power of two <= 32, aligned groups).
__device__ __forceinline__ void pair_reduce_lanes(float &h, float &l, int width)
{
    for (int o = width >> 1; o > 0; o >>= 1) {
        float bh = __shfl_xor_sync(0xffffffffu, h, o);
        float bl = __shfl_xor_sync(0xffffffffu, l, o);
        pair_add(h, l, bh, bl);
    }
}

// (h, l) += (bh, bl) without renormalisation (cascaded "Sum2"): the TwoSum
// error of the leading parts joins the trailing parts.  Symmetric in its two
// operands, so butterfly partners stay bit-identical.
__device__ __forceinline__ void pair_acc(float &h, float &l, float bh, float bl)
{
    float s, e;
    two_sum(h, bh, s, e);
    h = s;
    l = __fadd_rn(__fadd_rn(l, bl), e);
}

// Sum of the pairs (h, l) of the tpr threads of a multi-warp row group,
// returned to every thread of the group.  Every thread stores its pair; the
// first warp of the group adds the pairs of threads lane, lane+32, ... in
// that order, then the 32 lane sums in a butterfly, and publishes the total.
// red_h / red_l hold one slot per thread of the CTA, tot_h / tot_l one per
// group.  Two CTA barriers; the fixed order makes the result bitwise
// reproducible.
__device__ __forceinline__ void group_sum_pair(float &h, float &l, float *red_h, float *red_l,
                                               float *tot_h, float *tot_l, int grp, int tpr)
{
    red_h[threadIdx.x] = h;
    red_l[threadIdx.x] = l;
    __syncthreads();
    const int lane32 = threadIdx.x & 31;
    const int base = grp * tpr;
    if (threadIdx.x - base < 32) {
        h = red_h[base + lane32];
        l = red_l[base + lane32];
        for (int j = lane32 + 32; j < tpr; j += 32) pair_acc(h, l, red_h[base + j], red_l[base + j]);
        for (int o = 16; o > 0; o >>= 1) {
            const float bh = __shfl_xor_sync(0xffffffffu, h, o);
            const float bl = __shfl_xor_sync(0xffffffffu, l, o);
            pair_acc(h, l, bh, bl);
        }
        if (lane32 == 0) {
            tot_h[grp] = h;
            tot_l[grp] = l;
        }
    }
    __syncthreads();
    h = tot_h[grp];
    l = tot_l[grp];
}

}  // namespace crmsn
