// Short-sequence selective scan (L <= 4), the single-token recurrent step of inference above
// all: h = A_bar h + B_bar x, y = C.h + D x, times silu(z), the state advanced in place when
// h0 == h_last ("Mamba/SSM complete guide" section 2, recurrent inference with a constant-size
// state; section 5 `selective_scan` for the step itself).
//
// The step is bound by reading and writing the state (b, D, N) fp32 once. A group of N / 4
// threads owns one channel (b, d), each thread four consecutive states, so the state and the
// rows of A move as 16-byte loads and stores and a warp covers 512 contiguous bytes of each;
// the per-channel scalars (x, delta, z) and the per-token B, C rows are plain loads (B and C
// are shared by all channels and come from L1/L2). The group sums its readout with xor
// shuffles and its first thread finishes y. Arithmetic matches the generic kernel (CUDA's
// expf/log1pf softplus, expm1f for exact ZOH, an IEEE division in silu).
#include "common.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kDecodeThreads = 256;

template <int TPC>
__global__ void __launch_bounds__(kDecodeThreads) scan_decode_kernel(const ScanArgs a) {
    // Programmatic dependent launch: this grid may have started before the kernel ahead of it on
    // the stream finished (a decode loop's previous token, which wrote the state). Wait for that
    // grid's memory operations before the first global access, then let the next kernel's launch
    // begin while this one runs (it waits in turn). Without a programmatic predecessor the wait
    // returns at once. (Releasing the next launch before the wait, so that launches run two
    // steps ahead, measured 2.54 against 2.38 us per token.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t gtid = (int64_t)blockIdx.x * kDecodeThreads + threadIdx.x;
    const int64_t chan = gtid / TPC;
    const int g = (int)(gtid % TPC);
    const bool active = chan < a.batch * a.dim;   // whole groups are active or not
    const int64_t b = active ? chan / a.dim : 0;
    const int64_t d = active ? chan % a.dim : 0;
    const int N = a.dstate;
    const int n0 = 4 * g;

    float Av[4] = {0.f, 0.f, 0.f, 0.f}, h[4] = {0.f, 0.f, 0.f, 0.f};
    if (active && idx_ok(d * N + n0 + 3, a.dim * N, a.status)) {
        const float4 a4 = *reinterpret_cast<const float4*>(a.A + d * N + n0);
        Av[0] = a4.x;
        Av[1] = a4.y;
        Av[2] = a4.z;
        Av[3] = a4.w;
        if (a.h0 && idx_ok((b * a.dim + d) * N + n0 + 3, a.batch * a.dim * N, a.status)) {
            const float4 h4 = *reinterpret_cast<const float4*>(a.h0 + (b * a.dim + d) * N + n0);
            h[0] = h4.x;
            h[1] = h4.y;
            h[2] = h4.z;
            h[3] = h4.w;
        }
    }
    const float Dd = (active && a.D && idx_ok(d, a.dim, a.status)) ? a.D[d] : 0.f;
    const float bias = (active && a.bias && idx_ok(d, a.dim, a.status)) ? a.bias[d] : 0.f;

    for (int64_t step = 0; step < a.seqlen; ++step) {
        const int64_t t = a.reverse ? a.seqlen - 1 - step : step;
        float xv = 0.f, dv = 0.f, zv = 0.f, Bn[4] = {0.f, 0.f, 0.f, 0.f}, Cn[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
            const int64_t ix = b * a.xs[0] + t * a.xs[1] + d * a.xs[2];
            const int64_t id = b * a.ds[0] + t * a.ds[1] + d * a.ds[2];
            const int64_t iz = b * a.zs[0] + t * a.zs[1] + d * a.zs[2];
            if (idx_ok(ix, a.ext_x, a.status)) xv = load_f32(a.x, ix, a.io_bf16);
            if (idx_ok(id, a.ext_delta, a.status)) dv = load_f32(a.delta, id, a.io_bf16);
            if (a.z && idx_ok(iz, a.ext_z, a.status)) zv = load_f32(a.z, iz, a.io_bf16);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t ib = b * a.Bs[0] + t * a.Bs[1] + (n0 + k) * a.Bs[2];
                const int64_t ic = b * a.Cs[0] + t * a.Cs[1] + (n0 + k) * a.Cs[2];
                if (idx_ok(ib, a.ext_B, a.status)) Bn[k] = load_f32(a.B, ib, a.io_bf16);
                if (idx_ok(ic, a.ext_C, a.status)) Cn[k] = load_f32(a.C, ic, a.io_bf16);
            }
        }
        float dt = dv + bias;
        if (a.softplus) dt = softplus_accurate(dt);
        const float u = dt * xv;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float abar = ex2_approx(dt * Av[k] * kLog2e);
            const float bx = (a.zoh && Av[k] != 0.f) ? expm1f(dt * Av[k]) / Av[k] * Bn[k] * xv : u * Bn[k];
            h[k] = fmaf(abar, h[k], bx);
            acc = fmaf(Cn[k], h[k], acc);
        }
#pragma unroll
        for (int off = TPC / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (active && g == 0) {
            float out = fmaf(Dd, xv, acc);
            if (a.z) out *= silu_accurate(zv);
            const int64_t iy = b * a.ys[0] + t * a.ys[1] + d * a.ys[2];
            if (idx_ok(iy, a.ext_y, a.status)) store_io(a.y, iy, out, a.io_bf16);
        }
    }
    if (active && a.h_last && idx_ok((b * a.dim + d) * N + n0 + 3, a.batch * a.dim * N, a.status))
        *reinterpret_cast<float4*>(a.h_last + (b * a.dim + d) * N + n0) = make_float4(h[0], h[1], h[2], h[3]);
}

template <int TPC>
cudaError_t launch(const ScanArgs& a, cudaStream_t st) {
    const int64_t threads = a.batch * a.dim * TPC;
    const int64_t grid = (threads + kDecodeThreads - 1) / kDecodeThreads;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    // launched as a programmatic dependent of the previous kernel on the stream (see the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, scan_decode_kernel<TPC>, a);
    note_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool scan_decode_supported(const ScanArgs& a) {
    const int N = a.dstate;
    // N / 4 threads per channel: a power of two up to a warp, so groups never straddle warps
    if (N % 4 != 0 || N > 128 || ((N / 4) & (N / 4 - 1)) != 0 || a.conv_w) return false;
    if (!al16(a.A) || (a.h0 && !al16(a.h0)) || (a.h_last && !al16(a.h_last))) return false;
    return true;
}

cudaError_t launch_scan_decode(const ScanArgs& a, cudaStream_t st) {
    switch (a.dstate / 4) {
        case 1: return launch<1>(a, st);
        case 2: return launch<2>(a, st);
        case 4: return launch<4>(a, st);
        case 8: return launch<8>(a, st);
        case 16: return launch<16>(a, st);
        case 32: return launch<32>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssm
