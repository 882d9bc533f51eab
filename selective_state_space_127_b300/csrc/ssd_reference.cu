// SSD scan by the plain recurrence on CUDA cores: one CTA per (batch, head) walks the
// sequence with the N x P state spread over its threads. It is the general path for shapes
// the tensor-core chunked kernel does not take, and its results do not depend on the
// chunk length.
//
// Thread (p, j) of the CTA owns column p of the state for the rows n = j, j + J, j + 2J, ...
// Per step: dt = softplus(delta + bias); S[n][p] = exp(dt A_h) S[n][p] + dt B[n] x[p];
// the J partial sums of C[n] S[n][p] meet in shared memory.
//
// Recurrence: "Mamba-2 / Structured State Space Duality" (abeam) "基本アイデア"
// (h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t); "Mamba/SSM complete guide" section 6
// "SSD演算の概念" and `Mamba2Block` (one A per head).
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kRefThreads = 256;
constexpr int kRefMaxRows = 64;   // state rows per thread

__global__ void __launch_bounds__(kRefThreads)
ssd_reference_kernel(const SSDArgs a) {
    const int P = (int)a.headdim, N = (int)a.dstate;
    const int J = kRefThreads / P;                 // thread groups over the rows
    const int p = threadIdx.x % P, j = threadIdx.x / P;
    const bool active = j < J;
    const int64_t b = blockIdx.x / a.nheads, hh = blockIdx.x % a.nheads;
    const int64_t grp = hh / (a.nheads / a.ngroups);

    extern __shared__ float smem[];
    float* sB = smem;            // N
    float* sC = sB + N;          // N
    float* part = sC + N;        // J * P partial outputs

    float S[kRefMaxRows];
    const int rows = (N + J - 1) / J;
#pragma unroll
    for (int r = 0; r < kRefMaxRows; ++r) {
        const int n = j + r * J;
        S[r] = (active && r < rows && n < N && a.h0) ? a.h0[((b * a.nheads + hh) * N + n) * P + p] : 0.f;
    }
    const float Ah = a.A[hh] * kLog2e;
    const float bias = a.bias ? a.bias[hh] : 0.f;
    const float Dh = a.D ? a.D[hh] : 0.f;

    for (int64_t t = 0; t < a.seqlen; ++t) {
        const int64_t row = (b * a.seqlen + t) * a.ngroups + grp;
        for (int n = threadIdx.x; n < N; n += blockDim.x) {
            sB[n] = load_f32(a.B, row * N + n, a.io_bf16);
            sC[n] = load_f32(a.C, row * N + n, a.io_bf16);
        }
        float dt = load_f32(a.delta, (b * a.seqlen + t) * a.nheads + hh, a.io_bf16) + bias;
        if (a.softplus) dt = softplus_accurate(dt);
        const float abar = ex2_approx(dt * Ah);
        const int64_t xi = ((b * a.seqlen + t) * a.nheads + hh) * P + p;
        const float xv = active ? load_f32(a.x, xi, a.io_bf16) : 0.f;
        const float u = dt * xv;
        __syncthreads();
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < kRefMaxRows; ++r) {
            const int n = j + r * J;
            if (active && r < rows && n < N) {
                S[r] = fmaf(abar, S[r], u * sB[n]);
                acc = fmaf(sC[n], S[r], acc);
            }
        }
        if (active) part[j * P + p] = acc;
        __syncthreads();
        if (j == 0) {
            float out = 0.f;
            for (int q = 0; q < J; ++q) out += part[q * P + p];
            out = fmaf(Dh, xv, out);
            if (a.z) out *= silu_accurate(load_f32(a.z, xi, a.io_bf16));
            store_io(a.y, xi, out, a.io_bf16);
        }
        __syncthreads();
    }
    if (active && a.h_last) {
#pragma unroll
        for (int r = 0; r < kRefMaxRows; ++r) {
            const int n = j + r * J;
            if (r < rows && n < N) a.h_last[((b * a.nheads + hh) * N + n) * P + p] = S[r];
        }
    }
}

}  // namespace

// Valid for 1 <= P <= 256 and ceil(N / (256 / P)) <= 64 (the API layer checks this).
cudaError_t launch_ssd_reference(const SSDArgs& a, cudaStream_t st) {
    const int P = (int)a.headdim, N = (int)a.dstate;
    const int J = kRefThreads / P;
    const size_t smem = (size_t)(2 * N + J * P) * sizeof(float);
    ssd_reference_kernel<<<(unsigned)(a.batch * a.nheads), kRefThreads, smem, st>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
