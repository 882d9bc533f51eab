// Device helpers shared by the kernels: dtype conversion and fast transcendental forms.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssm {

// ---------------------------------------------------------------- index checks (debug build)
// A library compiled with -DSSM_DEBUG_CHECKS (`python -m selective_state_space_127_b300.build
// --debug-checks` -> libssmscan_debug.so) checks every computed global-memory index of its
// kernels against the extent of the array it addresses (TMA boxes are clipped by the hardware
// and need no check): an index outside latches SSM_ERR_BOUNDS in the call's status word and the
// access is skipped (a load reads zero). No trap, no fault. The normal build compiles the
// checks out.
#ifdef SSM_DEBUG_CHECKS
__device__ __forceinline__ bool idx_ok(int64_t i, int64_t n, unsigned* status) {
    if (i >= 0 && i < n) return true;
    if (status) atomicExch(status, 6u /* SSM_ERR_BOUNDS */);
    return false;
}
#else
__device__ __forceinline__ bool idx_ok(int64_t, int64_t, unsigned*) { return true; }
#endif

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

// silu(z) = z / (1 + 2^(-z log2 e)) with the SFU's ex2 and rcp (each about 1-2 ulp).
__device__ __forceinline__ float silu_fast(float z) { return z * rcp_approx(1.f + ex2_approx(-z * kLog2e)); }

}  // namespace ssm
