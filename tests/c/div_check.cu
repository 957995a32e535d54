// Bitwise check of the block quantiser's division by a scale (DivScale, five
// packed FMA-type instructions from the reciprocal) against CUDA's IEEE
// division __fdiv_rn, on pseudo-random dividends and divisors over wide
// exponent ranges plus the library's own divisors (0.04, 1, amax / 448).
// Within DivScale's stated domain (|v| >= 2^-96, a finite IEEE quotient) the
// quotients must be equal bit for bit; outside it, dividends below 2^-96 must
// give quotients below 2^-36 (FP8 zero).  Prints the number compared and the
// number of violations of each kind (both must be 0).
#include <cstdio>
#include <cstdint>

#include "common.cuh"

using namespace crmsn;

__device__ uint32_t mix(uint64_t x)   // SplitMix64 finaliser, low 32 bits
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)(x ^ (x >> 31));
}

// A float with a random 23-bit mantissa (or, with bf16 != 0, an 8-bit one)
// and an exponent uniform in [lo, hi].
__device__ float rnd(uint64_t key, int lo, int hi, int bf16)
{
    const uint32_t a = mix(key), b = mix(key ^ 0x5555);
    uint32_t m = a & 0x7FFFFF;
    if (bf16) m &= 0x7F0000;
    const int e = lo + (int)(b % (uint32_t)(hi - lo + 1));
    return __uint_as_float(((b >> 31) << 31) | ((uint32_t)(e + 127) << 23) | m);
}

__global__ void check(unsigned long long *normal_bad, unsigned long long *sub_bad,
                      unsigned long long *count)
{
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned long long nb = 0, sb = 0, n = 0;
    for (int it = 0; it < 64; ++it) {
        const uint64_t key = (tid * 64 + it) * 8;
        float s;
        switch (it & 3) {
            case 0: s = 0.04f; break;
            case 1: s = 1.0f; break;
            case 2: s = __fdiv_rn(rnd(key + 1, -20, 10, 1), 448.0f); break;   // amax / 448
            default: s = rnd(key + 1, -120, 120, 0); break;
        }
        const DivScale d(s);
        const int wide = (it >> 2) & 1;
        const float v0 = rnd(key + 2, wide ? -126 : -30, wide ? 127 : 30, it & 8);
        const float v1 = rnd(key + 3, wide ? -126 : -30, wide ? 127 : 30, it & 8);
        float q0, q1;
        d.div(f2(v0, v1), q0, q1);
        const float r0 = __fdiv_rn(v0, s), r1 = __fdiv_rn(v1, s);
        const float q[2] = {q0, q1}, r[2] = {r0, r1};
        const float v[2] = {v0, v1};
        for (int j = 0; j < 2; ++j) {
            if (!d.fast || !(fabsf(r[j]) <= 0x1.fffffep127f)) continue;   // IEEE path / overflow
            if (fabsf(v[j]) >= 0x1p-96f) {
                if (__float_as_uint(q[j]) != __float_as_uint(r[j])) ++nb;
            } else if (!(fabsf(q[j]) < 0x1p-36f)) {
                ++sb;
            }
        }
        n += 2;
    }
    atomicAdd(normal_bad, nb);
    atomicAdd(sub_bad, sb);
    atomicAdd(count, n);
}

int main()
{
    unsigned long long *d, h[3] = {0, 0, 0};
    if (cudaMalloc(&d, sizeof h) != cudaSuccess) return 2;
    cudaMemset(d, 0, sizeof h);
    check<<<2048, 256>>>(d, d + 1, d + 2);
    if (cudaMemcpy(h, d, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    cudaFree(d);
    printf("compared %llu mismatches %llu tiny_violations %llu\n", h[2], h[0], h[1]);
    return h[0] != 0 || h[1] != 0;
}
