// Device helpers shared by the kernels: dtype conversion and fast transcendental forms.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

__device__ __forceinline__ float load_f32(const void* p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_io(void* p, int64_t i, float v, int bf16) {
    if (bf16)
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else
        static_cast<float*>(p)[i] = v;
}

// 2^x with the SFU (ex2.approx.ftz.f32: relative error about 2^-22, flushes denormals).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) with the SFU.
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x with the SFU.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v) through CUDA's accurate expf/log1pf; v > 20 returns v
// (log1p(e^-v) < 2.1e-9 is below fp32 resolution there).
__device__ __forceinline__ float softplus_accurate(float v) {
    return v > 20.f ? v : log1pf(expf(v));
}

// silu(z) = z / (1 + e^-z) through CUDA's accurate expf and an IEEE division.
__device__ __forceinline__ float silu_accurate(float z) { return z / (1.f + expf(-z)); }

// softplus(v) = log(1 + e^v) from the SFU: e = 2^(v log2 e), then
//  * e < 1/16: the series log1p(e) = e - e^2/2 + ... - e^6/6 (truncation below 1e-8 relative),
//    which keeps full relative accuracy for the small steps (softplus near e^v);
//  * otherwise lg2(1 + e) ln 2 (SFU log error near 2^-22 absolute, < 2e-6 relative here);
//  * v > 15 returns v (the dropped log1p(e^-v) is below 2e-8 relative).
__device__ __forceinline__ float softplus_fast(float v) {
    const float e = ex2_approx(fminf(v, 15.f) * kLog2e);
    float s = fmaf(e, -1.f / 6.f, 0.2f);
    s = fmaf(e, s, -0.25f);
    s = fmaf(e, s, 1.f / 3.f);
    s = fmaf(e, s, -0.5f);
    s = fmaf(e, s, 1.f);
    const float series = e * s;
    const float lg = lg2_approx(1.f + e) * kLn2;
    const float r = e < 0.0625f ? series : lg;
    return v > 15.f ? v : r;
}

// silu(z) = z / (1 + 2^(-z log2 e)) with the SFU's ex2 and rcp (each about 1-2 ulp).
__device__ __forceinline__ float silu_fast(float z) { return z * rcp_approx(1.f + ex2_approx(-z * kLog2e)); }

}  // namespace ssm
