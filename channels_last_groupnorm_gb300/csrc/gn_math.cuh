// gn_math.cuh -- the arithmetic the GroupNorm kernel files share: packed
// fp32 pairs (the f32x2 instructions of sm_100+), the exact bf16 -> fp32
// widening, and the per-word apply y = x * scale + shift (+ SiLU).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "gn_ptx.cuh"

namespace gn {

typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t pk(float lo, float hi)
{
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void upk(f2_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f2_t add2(f2_t a, f2_t b)
{
    f2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2_t sub2(f2_t a, f2_t b)
{
    f2_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2_t mul2(f2_t a, f2_t b)
{
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c)
{
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// the two bf16 values packed in a 32-bit word, widened exactly to fp32
__device__ __forceinline__ f2_t bf2_to_f2(uint32_t w)
{
    return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// y = x * scale + shift (+ SiLU) for the two bf16 values of one word, on
// a packed pair: z = fma(x, s, t), then SiLU(z) = z * sigmoid(z) with
// sigmoid(z) = 1 / d, d = 1 + 2^(-z log2 e), from MUFU approximations (ex2,
// rcp; a few ulp of fp32).  A GB300 SM retires 32 ex2 but only 16
// reciprocals per clock, so the pair shares one reciprocal:
// 1/d0 = d1 / (d0 d1), 1/d1 = d0 / (d0 d1).  The exponent is capped at 63 so
// that d0 d1 stays finite (the cap moves sigmoid only where it is below
// 2^-63, i.e. z < -43, where the output rounds to zero anyway).
template <bool SILU>
__device__ __forceinline__ uint32_t apply_pair(uint32_t w, f2_t st_s, f2_t st_t)
{
    f2_t z = fma2(bf2_to_f2(w), st_s, st_t);
    if (SILU) {
        const f2_t arg = mul2(z, pk(-1.4426950408889634f, -1.4426950408889634f));
        float a0, a1;
        upk(arg, a0, a1);
        const f2_t den = add2(pk(ex2_approx(fminf(a0, 63.f)), ex2_approx(fminf(a1, 63.f))), pk(1.0f, 1.0f));
        float d0, d1;
        upk(den, d0, d1);
        const float r = rcp_approx(d0 * d1);
        z = mul2(mul2(z, pk(d1, d0)), pk(r, r));
    }
    float z0, z1;
    upk(z, z0, z1);
    const __nv_bfloat162 h = __floats2bfloat162_rn(z0, z1);
    return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace gn
