// Causal depthwise conv1d along t with K <= 4 taps per channel, then optionally SiLU: the
// prologue of the Mamba block's x branch,
//   v[b,t,d] = bias[d] + sum_k weight[d,k] * xp[b, t+k, d]  (xp = x_prev then x along t),
//   y = silu(v) or v.
// Pages: "Mamba/SSM complete guide" section 5 `MambaBlock` (depthwise nn.Conv1d, kernel
// d_conv, padding d_conv - 1, output cut to the first L steps, then F.silu); "論文解説: Mamba"
// "Mambaブロックの全体構成" (a d_conv = 4 convolution followed by SiLU).
//
// The operation reads x once and writes y once, so it is bound by HBM bandwidth. Each thread
// owns four channels (8 bytes of bf16, 16 of fp32) and a run of kRun consecutive steps: it keeps
// the K-1 previous inputs of its channels in registers and walks the run in groups of kSub
// rows, issuing a group's loads (read-only path) before its arithmetic. Four channels keep the
// thread within 80 registers, so 24 warps per SM keep 37 KB (bf16) to 74 KB (fp32) of loads in
// flight. Consecutive threads take consecutive channel groups of one (b, run), so a warp reads and
// writes 256 (bf16) or 512 (fp32) contiguous bytes per step. The K-1 rows before a run are read
// a second time (by the run that owns them), from L2.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 256;
constexpr int kRun = 36;   // steps per thread (six groups)
constexpr int kSub = 6;    // rows loaded ahead of their arithmetic

template <bool BF16>
struct Vec;
// Four channels of one row: the raw load, its widening to fp32, and the rounded store.
template <>
struct Vec<true> {
    static constexpr int kN = 4;
    using Raw = uint2;
    static __device__ __forceinline__ Raw load(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
    static __device__ __forceinline__ void widen(Raw q, float (&v)[4]) {
        v[0] = __uint_as_float(q.x << 16);
        v[1] = __uint_as_float(q.x & 0xffff0000u);
        v[2] = __uint_as_float(q.y << 16);
        v[3] = __uint_as_float(q.y & 0xffff0000u);
    }
    static __device__ __forceinline__ void store(void* p, const float (&v)[4]) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2*>(p) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
};
template <>
struct Vec<false> {
    static constexpr int kN = 4;
    using Raw = float4;
    static __device__ __forceinline__ Raw load(const void* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
    static __device__ __forceinline__ void widen(Raw q, float (&v)[4]) {
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    }
    static __device__ __forceinline__ void store(void* p, const float (&v)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

template <bool BF16, int K, bool SILU>
__global__ void __launch_bounds__(kConvThreads, 3)
conv1d_kernel(const void* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
              const void* __restrict__ x_prev, void* __restrict__ y, int64_t batch, int64_t L, int64_t dim) {
    using V = Vec<BF16>;
    constexpr int E = V::kN;                 // channels per thread
    constexpr int64_t kEsz = BF16 ? 2 : 4;
    const int64_t ng = dim / E;              // channel groups
    const int64_t nruns = (L + kRun - 1) / kRun;
    const int64_t item = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
    if (item >= batch * nruns * ng) return;
    const int64_t cg = item % ng;
    const int64_t run = (item / ng) % nruns;
    const int64_t b = item / (ng * nruns);
    const int64_t d0 = cg * E;
    const int64_t t0 = run * kRun;
    const char* xb = static_cast<const char*>(x) + (b * L * dim + d0) * kEsz;
    char* yb = static_cast<char*>(y) + (b * L * dim + d0) * kEsz;

    float wk[K][E], bv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        bv[e] = bias ? bias[d0 + e] : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) wk[k][e] = w[(d0 + e) * K + k];
    }
    // win[j] holds x_{t-(K-1)+j} for j < K-1 before step t
    float win[K > 1 ? K - 1 : 1][E];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t tt = t0 - (K - 1) + j;
        if (tt >= 0) {
            V::widen(V::load(xb + tt * dim * kEsz), win[j]);
        } else if (x_prev) {
            // x_prev[b, K-1+tt, :] is x_{tt}
            V::widen(V::load(static_cast<const char*>(x_prev) + ((b * (K - 1) + (K - 1) + tt) * dim + d0) * kEsz),
                     win[j]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) win[j][e] = 0.f;
        }
    }
    const int nt = (int)(L - t0 < kRun ? L - t0 : kRun);
#pragma unroll 1
    for (int i0 = 0; i0 < nt; i0 += kSub) {
        typename V::Raw raw[kSub];
#pragma unroll
        for (int i = 0; i < kSub; ++i)
            if (i0 + i < nt) raw[i] = V::load(xb + (t0 + i0 + i) * dim * kEsz);
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            if (i0 + i < nt) {
                float xv[E], out[E];
                V::widen(raw[i], xv);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    float v = fmaf(wk[K - 1][e], xv[e], bv[e]);
#pragma unroll
                    for (int j = 0; j < K - 1; ++j) v = fmaf(wk[j][e], win[j][e], v);
                    // silu from the SFU's ex2 and rcp (a few ulp): the kernel stays bound by
                    // memory, not by instruction issue
                    out[e] = SILU ? silu_fast(v) : v;
                }
                V::store(yb + (t0 + i0 + i) * dim * kEsz, out);
                // slide the window
#pragma unroll
                for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
                    for (int e = 0; e < E; ++e) win[j][e] = win[j + 1][e];
                if constexpr (K > 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) win[K - 2][e] = xv[e];
                }
            }
        }
    }
}

template <bool BF16, int K>
cudaError_t launch_k(const Conv1dArgs& a, cudaStream_t st) {
    constexpr int E = Vec<BF16>::kN;
    const int64_t items = a.batch * ((a.seqlen + kRun - 1) / kRun) * (a.dim / E);
    const int64_t grid = (items + kConvThreads - 1) / kConvThreads;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    if (a.silu)
        conv1d_kernel<BF16, K, true><<<(unsigned)grid, kConvThreads, 0, st>>>(a.x, a.w, a.bias, a.x_prev, a.y,
                                                                              a.batch, a.seqlen, a.dim);
    else
        conv1d_kernel<BF16, K, false><<<(unsigned)grid, kConvThreads, 0, st>>>(a.x, a.w, a.bias, a.x_prev, a.y,
                                                                               a.batch, a.seqlen, a.dim);
    note_launches(1);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_t(const Conv1dArgs& a, cudaStream_t st) {
    switch (a.k) {
        case 1: return launch_k<BF16, 1>(a, st);
        case 2: return launch_k<BF16, 2>(a, st);
        case 3: return launch_k<BF16, 3>(a, st);
        case 4: return launch_k<BF16, 4>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_conv1d(const Conv1dArgs& a, cudaStream_t st) {
    return a.io_bf16 ? launch_t<true>(a, st) : launch_t<false>(a, st);
}

}  // namespace ssm
