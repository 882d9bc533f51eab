// SSD scan by the plain recurrence on CUDA cores: one CTA per (batch, head) walks the
// sequence with the N x P state spread over its threads. It is the general path for shapes
// and dtypes the tensor-core chunked kernel does not take (any P <= 256, any N the state fits,
// fp32 I/O), and its results do not depend on the chunk length.
//
// Thread (p, j) of the CTA owns column p of the state for the rows n = j rows .. (j + 1) rows - 1
// (rows = ceil(N / J)), so it reads the B and C values of its rows as 16-byte vectors (the
// whole warp reads the same ones: a broadcast).
// The sequence goes in tiles of kT steps: the CTA stages the tile's B and C rows, x rows and
// dt = softplus(delta + bias) in shared memory with coalesced loads, then every thread runs the
// kT steps on its state rows,
//   S[n][p] = exp(dt A_h) S[n][p] + dt B[n] x[p],   part_t = sum over its rows of C[n] S[n][p],
// writing each step's partial readout to shared memory; the J partial sums of each (t, p) are
// added once per tile, and y leaves with coalesced stores. Three barriers per tile instead of
// three per step.
//
// Recurrence: "Mamba-2 / Structured State Space Duality" (abeam) "基本アイデア"
// (h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t); "Mamba/SSM complete guide" section 6
// "SSD演算の概念" and `Mamba2Block` (one A per head).
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kRefThreads = 256;
constexpr int kRefMaxRows = 64;   // state rows per thread at most
constexpr int kT = 32;            // steps per tile

// ROWS: the state rows a thread keeps (a power of two >= ceil(N / J)); VEC: rows is a multiple
// of 4 and J rows == N, so a thread's B and C values are 16-byte aligned runs.
template <int ROWS, bool VEC>
__global__ void __launch_bounds__(kRefThreads, ROWS >= 64 ? 1 : 2)
ssd_reference_kernel(const SSDArgs a) {
    const int P = (int)a.headdim, N = (int)a.dstate;
    const int J = kRefThreads / P;                 // thread groups over the rows
    const int p = threadIdx.x % P, j = threadIdx.x / P;
    const bool active = j < J;
    const int64_t b = blockIdx.x / a.nheads, hh = blockIdx.x % a.nheads;
    const int64_t grp = hh / (a.nheads / a.ngroups);
    const int tid = threadIdx.x;

    extern __shared__ float smem[];
    float* sB = smem;                 // [kT][N]
    float* sC = sB + kT * N;          // [kT][N]
    float* sx = sC + kT * N;          // [kT][P]
    float* sdt = sx + kT * P;         // [kT]
    float* part = sdt + kT;           // [J][kT][P] partial readouts

    float S[ROWS];
    const int rows = (N + J - 1) / J;
    // extents for the index checks of the debug build
    const int64_t n_state = a.batch * a.nheads * N * P, n_act = a.batch * a.seqlen * a.nheads * P;
    const int64_t n_bc = a.batch * a.seqlen * a.ngroups * N, n_dt = a.batch * a.seqlen * a.nheads;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int n = j * rows + r;
        const int64_t is = ((b * a.nheads + hh) * N + n) * P + p;
        S[r] = (active && r < rows && n < N && a.h0 && idx_ok(is, n_state, a.status)) ? a.h0[is] : 0.f;
    }
    const float Ah = a.A[hh] * kLog2e;
    const float bias = a.bias ? a.bias[hh] : 0.f;
    const float Dh = a.D ? a.D[hh] : 0.f;

    for (int64_t t0 = 0; t0 < a.seqlen; t0 += kT) {
        const int nt = (int)(a.seqlen - t0 < kT ? a.seqlen - t0 : kT);
        // ---- stage the tile
        for (int i = tid; i < nt * N; i += kRefThreads) {
            const int tt = i / N, n = i % N;
            const int64_t row = (b * a.seqlen + t0 + tt) * a.ngroups + grp;
            const bool okb = idx_ok(row * N + n, n_bc, a.status);
            sB[tt * N + n] = okb ? load_f32(a.B, row * N + n, a.io_bf16) : 0.f;
            sC[tt * N + n] = okb ? load_f32(a.C, row * N + n, a.io_bf16) : 0.f;
        }
        for (int i = tid; i < nt * P; i += kRefThreads) {
            const int tt = i / P, q = i % P;
            const int64_t ix = ((b * a.seqlen + t0 + tt) * a.nheads + hh) * P + q;
            sx[tt * P + q] = idx_ok(ix, n_act, a.status) ? load_f32(a.x, ix, a.io_bf16) : 0.f;
        }
        if (tid < kT) {
            float dt = 0.f;
            const int64_t id = (b * a.seqlen + t0 + tid) * a.nheads + hh;
            if (tid < nt && idx_ok(id, n_dt, a.status)) {
                dt = load_f32(a.delta, id, a.io_bf16) + bias;
                if (a.softplus) dt = softplus_accurate(dt);
            }
            sdt[tid] = dt;
        }
        __syncthreads();
        // ---- the tile's steps on this thread's state rows; each step's partial readout goes
        // to shared memory
        if (active) {
            for (int tt = 0; tt < nt; ++tt) {
                const float dt = sdt[tt];
                const float abar = ex2_approx(dt * Ah);
                const float u = dt * sx[tt * P + p];
                const float* bt = sB + tt * N + j * rows;
                const float* ct = sC + tt * N + j * rows;
                float s = 0.f;
                if constexpr (VEC) {
#pragma unroll
                    for (int r = 0; r < ROWS; r += 4) {
                        if (r < rows) {
                            const float4 b4 = *reinterpret_cast<const float4*>(bt + r);
                            const float4 c4 = *reinterpret_cast<const float4*>(ct + r);
                            S[r] = fmaf(abar, S[r], u * b4.x);
                            s = fmaf(c4.x, S[r], s);
                            S[r + 1] = fmaf(abar, S[r + 1], u * b4.y);
                            s = fmaf(c4.y, S[r + 1], s);
                            S[r + 2] = fmaf(abar, S[r + 2], u * b4.z);
                            s = fmaf(c4.z, S[r + 2], s);
                            S[r + 3] = fmaf(abar, S[r + 3], u * b4.w);
                            s = fmaf(c4.w, S[r + 3], s);
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        if (r < rows && j * rows + r < N) {
                            S[r] = fmaf(abar, S[r], u * bt[r]);
                            s = fmaf(ct[r], S[r], s);
                        }
                    }
                }
                part[(j * kT + tt) * P + p] = s;
            }
        }
        __syncthreads();
        // ---- y of the tile: sum the J partials, D skip, gate
        for (int i = tid; i < nt * P; i += kRefThreads) {
            const int tt = i / P, q = i % P;
            float out = 0.f;
            for (int g = 0; g < J; ++g) out += part[(g * kT + tt) * P + q];
            out = fmaf(Dh, sx[tt * P + q], out);
            const int64_t xi = ((b * a.seqlen + t0 + tt) * a.nheads + hh) * P + q;
            if (!idx_ok(xi, n_act, a.status)) continue;
            if (a.z) out *= silu_accurate(load_f32(a.z, xi, a.io_bf16));
            store_io(a.y, xi, out, a.io_bf16);
        }
        __syncthreads();
    }
    if (active && a.h_last) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int n = j * rows + r;
            const int64_t is = ((b * a.nheads + hh) * N + n) * P + p;
            if (r < rows && n < N && idx_ok(is, n_state, a.status)) a.h_last[is] = S[r];
        }
    }
}

}  // namespace

// Valid for 1 <= P <= 256 and ceil(N / (256 / P)) <= 64 (the API layer checks this).
cudaError_t launch_ssd_reference(const SSDArgs& a, cudaStream_t st) {
    const int P = (int)a.headdim, N = (int)a.dstate;
    const int J = kRefThreads / P;
    const size_t smem = (size_t)(2 * kT * N + kT * P + kT + J * kT * P) * sizeof(float);
    const int rows = (N + J - 1) / J;
    const bool vec = rows % 4 == 0 && rows * J == N;
    auto kern = rows <= 8 ? (vec ? ssd_reference_kernel<8, true> : ssd_reference_kernel<8, false>)
              : rows <= 16 ? (vec ? ssd_reference_kernel<16, true> : ssd_reference_kernel<16, false>)
              : rows <= 32 ? (vec ? ssd_reference_kernel<32, true> : ssd_reference_kernel<32, false>)
                           : (vec ? ssd_reference_kernel<kRefMaxRows, true> : ssd_reference_kernel<kRefMaxRows, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(a.batch * a.nheads), kRefThreads, smem, st>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
