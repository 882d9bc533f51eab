// Generic selective-scan kernel: any element strides (including broadcast), fp32 or bf16
// I/O, N up to 256, forward or reverse, delta*B or exact-ZOH discretisation.
//
// One channel (b, d) is a group of G consecutive lanes of a warp; lane g of the group
// keeps the fp32 states n in [g*S, g*S + S) in registers and walks the whole sequence.
// Per step each lane forms A_bar = 2^(dt * A * log2 e) for its states, updates them and
// accumulates its part of C.h; the group sums the parts with butterfly shuffles and its
// first lane adds D x, applies the silu(z) gate and stores y.
//
// Recurrence: "Mamba/SSM complete guide" section 5 `selective_scan` (deltaA = exp(delta A),
// deltaB_u = delta B u, x = deltaA x + deltaB_u, y = x.C, y + u D) and MambaBlock.forward
// (y * silu(z)); "論文解説: Mamba" "選択機構" (softplus) and "Hardware-Aware Parallel Scan".
// Exact ZOH: "State Space Model / Mamba" "Zero-Order Hold", `discretize_zoh`.
// Optional prologue: x replaced by silu(causal depthwise conv1d(x)) with a window of the
// K - 1 previous raw inputs in registers ("Mamba/SSM complete guide" section 5 `MambaBlock`:
// conv1d with padding d_conv - 1 cut to L steps, then F.silu).
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kGenericThreads = 128;

template <int S, int G>
__global__ void __launch_bounds__(kGenericThreads)
scan_generic_kernel(const ScanArgs a) {
    const int g = threadIdx.x % G;
    const int64_t chan = (int64_t)blockIdx.x * (kGenericThreads / G) + threadIdx.x / G;
    const bool active = chan < a.batch * a.dim;
    const int64_t b = active ? chan / a.dim : 0;
    const int64_t d = active ? chan % a.dim : 0;
    const int N = a.dstate;
    const int n0 = g * S;

    float A2[S], Araw[S], h[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int n = n0 + s;
        const bool ok = active && n < N;
        Araw[s] = ok && idx_ok(d * N + n, a.dim * N, a.status) ? a.A[d * N + n] : 0.f;
        A2[s] = Araw[s] * kLog2e;
        h[s] = (ok && a.h0 && idx_ok((b * a.dim + d) * N + n, a.batch * a.dim * N, a.status))
                   ? a.h0[(b * a.dim + d) * N + n]
                   : 0.f;
    }
    const float Dd = (active && a.D && idx_ok(d, a.dim, a.status)) ? a.D[d] : 0.f;
    const float bias = (active && a.bias && idx_ok(d, a.dim, a.status)) ? a.bias[d] : 0.f;
    // conv prologue: taps right-aligned into cw[0..3] (cw[3] multiplies x_t), win = x_{t-3..t-1}
    float cw[4] = {0.f, 0.f, 0.f, 0.f}, cb = 0.f, win[3] = {0.f, 0.f, 0.f};
    if (a.conv_w && active) {
        const int K = a.conv_k;
        for (int j = 4 - K; j < 4; ++j)
            if (idx_ok(d * K + j - (4 - K), a.dim * K, a.status)) cw[j] = a.conv_w[d * K + j - (4 - K)];
        cb = a.conv_b ? a.conv_b[d] : 0.f;
        if (a.conv_prev)
            for (int m = 1; m < K; ++m) {   // x_{-m} = x_prev[b, K-1-m]
                const int64_t i = (b * (K - 1) + (K - 1 - m)) * a.dim + d;
                if (idx_ok(i, a.batch * (K - 1) * a.dim, a.status)) win[3 - m] = load_f32(a.conv_prev, i, a.io_bf16);
            }
    }

    for (int64_t step = 0; step < a.seqlen; ++step) {
        const int64_t t = a.reverse ? a.seqlen - 1 - step : step;
        float xv = 0.f, dv = 0.f, zv = 0.f;
        if (active) {
            const int64_t ix = b * a.xs[0] + t * a.xs[1] + d * a.xs[2];
            const int64_t id = b * a.ds[0] + t * a.ds[1] + d * a.ds[2];
            const int64_t iz = b * a.zs[0] + t * a.zs[1] + d * a.zs[2];
            if (idx_ok(ix, a.ext_x, a.status)) xv = load_f32(a.x, ix, a.io_bf16);
            if (idx_ok(id, a.ext_delta, a.status)) dv = load_f32(a.delta, id, a.io_bf16);
            if (a.z && idx_ok(iz, a.ext_z, a.status)) zv = load_f32(a.z, iz, a.io_bf16);
        }
        if (a.conv_w) {
            const float v = fmaf(cw[3], xv, fmaf(cw[2], win[2], fmaf(cw[1], win[1], fmaf(cw[0], win[0], cb))));
            win[0] = win[1];
            win[1] = win[2];
            win[2] = xv;
            xv = silu_accurate(v);
        }
        float dt = dv + bias;
        if (a.softplus) dt = softplus_accurate(dt);
        const float u = dt * xv;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int n = n0 + s;
            if (active && n < N) {
                const int64_t ib = b * a.Bs[0] + t * a.Bs[1] + n * a.Bs[2];
                const int64_t ic = b * a.Cs[0] + t * a.Cs[1] + n * a.Cs[2];
                const float Bn = idx_ok(ib, a.ext_B, a.status) ? load_f32(a.B, ib, a.io_bf16) : 0.f;
                const float Cn = idx_ok(ic, a.ext_C, a.status) ? load_f32(a.C, ic, a.io_bf16) : 0.f;
                const float abar = ex2_approx(dt * A2[s]);
                float bx;
                if (a.zoh && Araw[s] != 0.f)
                    bx = expm1f(dt * Araw[s]) / Araw[s] * Bn * xv;
                else
                    bx = u * Bn;
                h[s] = fmaf(abar, h[s], bx);
                acc = fmaf(Cn, h[s], acc);
            }
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (active && g == 0) {
            float out = fmaf(Dd, xv, acc);
            if (a.z) out *= silu_accurate(zv);
            const int64_t iy = b * a.ys[0] + t * a.ys[1] + d * a.ys[2];
            if (idx_ok(iy, a.ext_y, a.status)) store_io(a.y, iy, out, a.io_bf16);
        }
    }
    if (active && a.h_last) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int n = n0 + s;
            if (n < N && idx_ok((b * a.dim + d) * N + n, a.batch * a.dim * N, a.status))
                a.h_last[(b * a.dim + d) * N + n] = h[s];
        }
    }
}

template <int S, int G>
cudaError_t launch(const ScanArgs& a, cudaStream_t st) {
    const int64_t nchan = a.batch * a.dim;
    const int64_t per_block = kGenericThreads / G;
    const int64_t grid = (nchan + per_block - 1) / per_block;
    scan_generic_kernel<S, G><<<(unsigned)grid, kGenericThreads, 0, st>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_generic(const ScanArgs& a, cudaStream_t st) {
    const int N = a.dstate;
    if (N <= 4) return launch<4, 1>(a, st);
    if (N <= 8) return launch<8, 1>(a, st);
    if (N <= 16) return launch<8, 2>(a, st);
    if (N <= 32) return launch<8, 4>(a, st);
    if (N <= 64) return launch<16, 4>(a, st);
    if (N <= 128) return launch<16, 8>(a, st);
    return launch<16, 16>(a, st);
}

}  // namespace ssm
