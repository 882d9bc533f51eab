// Unit-rate microbenchmark of one B300 SM: the per-clock throughput of the instructions the
// selective scan's state update is built from (SFU ex2 / lg2 / rcp / tanh, FP32 FMA scalar and
// packed f32x2, shared-memory loads by width and sharing pattern, warp shuffles, legacy
// mma.sync). These rates set the "alu" roofline the benchmark reports for the scan:
// one state update needs one ex2 and four FP32 lane operations, and its B and C values come
// out of shared memory.
//
// Method: one CTA of 512 threads per SM (148 CTAs), every thread issuing a long unrolled run
// of independent instances of one instruction (inline asm volatile, so nothing is folded or
// hoisted); thread 0 reads clock64 around the run after a barrier, so the rate is
//     lane operations / SM cycles
// averaged over the CTAs. Shared-memory loads are reported as bytes delivered to registers
// per clock and as wavefronts per warp instruction implied by that rate.
//
// Build and run: python -m selective_state_space_127_b300.unit_rates  (prints one JSON object)
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

constexpr int kThreads = 512;
constexpr int kIters = 256;
constexpr int kUnroll = 16;

struct Sample {
    unsigned long long cycles;
};

__device__ __forceinline__ void start_clock(unsigned long long& t0) {
    __syncthreads();
    t0 = clock64();
}

__device__ __forceinline__ void stop_clock(unsigned long long t0, Sample* out) {
    __syncthreads();
    if (threadIdx.x == 0) out[blockIdx.x].cycles = clock64() - t0;
}

// ---------------------------------------------------------------- SFU and FMA

template <int OP>
__global__ void __launch_bounds__(kThreads, 1) k_alu(float seed, Sample* out, float* sink) {
    float v[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) v[i] = seed * (0.25f + 0.01f * i) - 0.5f;
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            float r;
            if constexpr (OP == 0) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v[i]));
            if constexpr (OP == 1) asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v[i]));
            // rcp and tanh chains take an added constant (an FP32 add beside each SFU op), so
            // that nothing folds two applications into one
            if constexpr (OP == 2) asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v[i] + 1.5f));
            if constexpr (OP == 3) asm volatile("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v[i] + 0.5f));
            if constexpr (OP == 4) asm volatile("fma.rn.f32 %0, %1, %1, %1;" : "=f"(r) : "f"(v[i]));
            v[i] = r;
        }
    }
    stop_clock(t0, out);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) s += v[i];
    if (s == 123.456f) *sink = s;
}

// packed pairs: fma.rn.f32x2 (two lane operations per thread instruction)
__global__ void __launch_bounds__(kThreads, 1) k_fma2(float seed, Sample* out, float* sink) {
    unsigned long long v[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        float a = seed * 0.5f + i, b = seed * 0.25f - i;
        asm("mov.b64 %0, {%1, %2};" : "=l"(v[i]) : "f"(a), "f"(b));
    }
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) asm volatile("fma.rn.f32x2 %0, %0, %0, %0;" : "+l"(v[i]));
    }
    stop_clock(t0, out);
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) s ^= v[i];
    if (s == 12345ull) *sink = 1.f;
}

// one ex2 and two packed FP32 pairs per thread and step, the instruction mix of two state updates
__global__ void __launch_bounds__(kThreads, 1) k_mix(float seed, Sample* out, float* sink) {
    float e[kUnroll];
    unsigned long long p[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        e[i] = seed - i * 0.01f;
        float a = seed * 0.5f + i, b = seed * 0.25f - i;
        asm("mov.b64 %0, {%1, %2};" : "=l"(p[i]) : "f"(a), "f"(b));
    }
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            float r;
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e[i]));
            e[i] = r;
            asm volatile("fma.rn.f32x2 %0, %0, %0, %0;" : "+l"(p[i]));
            asm volatile("fma.rn.f32x2 %0, %0, %0, %0;" : "+l"(p[i]));
        }
    }
    stop_clock(t0, out);
    float s = 0.f;
    unsigned long long q = 0;
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        s += e[i];
        q ^= p[i];
    }
    if (s == 123.456f || q == 12345ull) *sink = s;
}

// ---------------------------------------------------------------- shared memory and shuffles

// Loads are volatile so that repeated addresses are not merged. MODE 0: every lane reads the same 16 bytes; 1: two addresses (lanes by parity of lane / 16);
// 2: 16-byte chunks distinct per lane (512 contiguous bytes per warp); 3: 4-byte broadcast;
// 4: 8-byte loads, two addresses.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_lds(Sample* out, float* sink) {
    __shared__ __align__(16) float buf[4096];
    for (int i = threadIdx.x; i < 4096; i += kThreads) buf[i] = (float)i;
    const int lane = threadIdx.x & 31;
    int off;   // float offset
    if (MODE == 0 || MODE == 3) off = 0;
    else if (MODE == 1 || MODE == 4) off = (lane >> 4) * 4;
    else off = lane * 4;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(buf + off);
    uint32_t acc = 0;   // every loaded word is folded in (integer xor, off the FP32 pipe)
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const uint32_t a = base + (uint32_t)((i & 3) * 2048) + (acc & 0u);
            if constexpr (MODE <= 2) {
                uint32_t x, y, z, w;
                asm volatile("ld.volatile.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "r"(a));
                acc ^= x ^ y ^ z ^ w;
            } else if constexpr (MODE == 3) {
                uint32_t x;
                asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(x) : "r"(a));
                acc ^= x;
            } else {
                uint32_t x, y;
                asm volatile("ld.volatile.shared.v2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
                acc ^= x ^ y;
            }
        }
    }
    stop_clock(t0, out);
    if (acc == 0x12345u) *sink = 1.f;
}

__global__ void __launch_bounds__(kThreads, 1) k_shfl(Sample* out, float* sink) {
    float v[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) v[i] = threadIdx.x + i;
    const int src = (threadIdx.x * 7 + 3) & 31;   // a runtime source lane
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            float r;
            asm volatile("shfl.sync.idx.b32 %0, %1, %2, 0x1f, 0xffffffff;" : "=f"(r) : "f"(v[i]), "r"(src ^ i));
            v[i] = r;
        }
    }
    stop_clock(t0, out);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) s += v[i];
    if (s == 123.456f) *sink = s;
}

// ---------------------------------------------------------------- legacy warp MMA

// KIND 0: mma.sync m16n8k8 tf32 -> f32; 1: m16n8k16 bf16 -> f32. Four independent accumulators.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) k_mma(Sample* out, float* sink) {
    float d[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[j][i] = 0.f;
    const uint32_t a0 = 0x3f800000u + threadIdx.x, a1 = 0x3f000000u, a2 = 0x3e800000u, a3 = 0x3f400000u;
    const uint32_t b0 = 0x3f800000u, b1 = 0x3f000000u + threadIdx.x;
    unsigned long long t0;
    start_clock(t0);
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int u = 0; u < kUnroll / 4; ++u) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (KIND == 0)
                    asm volatile(
                        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                        "{%0,%1,%2,%3};"
                        : "+f"(d[j][0]), "+f"(d[j][1]), "+f"(d[j][2]), "+f"(d[j][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                else
                    asm volatile(
                        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                        "{%8,%9}, {%0,%1,%2,%3};"
                        : "+f"(d[j][0]), "+f"(d[j][1]), "+f"(d[j][2]), "+f"(d[j][3])
                        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            }
        }
    }
    stop_clock(t0, out);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) s += d[j][i];
    if (s == 123.456f) *sink = s;
}

// ---------------------------------------------------------------- state-update loops

// The selective scan's state update with its operands in registers: per step and state
//   A_bar = 2^(dt a_n);  h_n = A_bar h_n + u b_n;  acc += c_n h_n
// for S states per thread, the step scalars dt, u changing every step. PACKED uses the
// f32x2 forms for the four FP32 operations. Reports updates per clock per SM.
template <bool PACKED, int S>
__global__ void k_update(float seed, Sample* out, float* sink, int steps) {
    float a[S], b[S], c[S], h[S];
#pragma unroll
    for (int n = 0; n < S; ++n) {
        a[n] = -(n + 1) * 1.4426950408889634f;
        b[n] = 0.5f + 0.01f * n;
        c[n] = 0.25f - 0.01f * n;
        h[n] = 0.f;
    }
    float dt = 0.01f + seed * 1e-3f, u = 0.3f;
    float acc = 0.f;
    unsigned long long t0;
    start_clock(t0);
    for (int t = 0; t < steps; ++t) {
        dt = fmaf(dt, 0.9999f, 1e-7f);
        u = fmaf(u, 0.9993f, 1e-6f);
        if constexpr (PACKED) {
            unsigned long long dt2, u2, acc2;
            asm("mov.b64 %0, {%1, %1};" : "=l"(dt2) : "f"(dt));
            asm("mov.b64 %0, {%1, %1};" : "=l"(u2) : "f"(u));
            asm("mov.b64 %0, {%1, %1};" : "=l"(acc2) : "f"(0.f));
#pragma unroll
            for (int n = 0; n < S; n += 2) {
                unsigned long long a2, b2, c2, h2, e2, ab2, ub2;
                asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "f"(a[n]), "f"(a[n + 1]));
                asm("mov.b64 %0, {%1, %2};" : "=l"(b2) : "f"(b[n]), "f"(b[n + 1]));
                asm("mov.b64 %0, {%1, %2};" : "=l"(c2) : "f"(c[n]), "f"(c[n + 1]));
                asm("mov.b64 %0, {%1, %2};" : "=l"(h2) : "f"(h[n]), "f"(h[n + 1]));
                asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(e2) : "l"(dt2), "l"(a2));
                float e0, e1, x0, x1;
                asm("mov.b64 {%0, %1}, %2;" : "=f"(e0), "=f"(e1) : "l"(e2));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x0) : "f"(e0));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x1) : "f"(e1));
                asm("mov.b64 %0, {%1, %2};" : "=l"(ab2) : "f"(x0), "f"(x1));
                asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(ub2) : "l"(u2), "l"(b2));
                asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(h2) : "l"(ab2), "l"(h2), "l"(ub2));
                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(c2), "l"(h2));
                asm("mov.b64 {%0, %1}, %2;" : "=f"(h[n]), "=f"(h[n + 1]) : "l"(h2));
            }
            float lo, hi;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc2));
            acc += lo + hi;
        } else {
            float s = 0.f;
#pragma unroll
            for (int n = 0; n < S; ++n) {
                float ab;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ab) : "f"(dt * a[n]));
                h[n] = fmaf(ab, h[n], u * b[n]);
                s = fmaf(c[n], h[n], s);
            }
            acc += s;
        }
    }
    stop_clock(t0, out);
    if (acc == 123.456f) *sink = acc;
}

// ---------------------------------------------------------------- host

int g_sms = 0;
Sample* g_out = nullptr;
float* g_sink = nullptr;

template <typename F>
double run(F launch, double* mhz) {
    launch();   // warm-up
    cudaDeviceSynchronize();
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventRecord(e0);
    launch();
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    Sample* h = new Sample[g_sms];
    cudaMemcpy(h, g_out, sizeof(Sample) * g_sms, cudaMemcpyDeviceToHost);
    double cyc = 0;
    unsigned long long mx = 0;
    for (int i = 0; i < g_sms; ++i) {
        cyc += (double)h[i].cycles;
        if (h[i].cycles > mx) mx = h[i].cycles;
    }
    delete[] h;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (mhz) *mhz = (double)mx / (ms * 1e3);
    return cyc / g_sms;   // mean SM cycles of the timed run
}

}  // namespace

int main() {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, 0) != cudaSuccess) {
        printf("{\"error\": \"no CUDA device\"}\n");
        return 1;
    }
    g_sms = prop.multiProcessorCount;
    cudaMalloc(&g_out, sizeof(Sample) * g_sms);
    cudaMalloc(&g_sink, sizeof(float));
    const double per_thread = (double)kIters * kUnroll;
    const double lanes = (double)kThreads * per_thread;   // lane operations per SM
    const dim3 grid(g_sms), block(kThreads);
    double mhz = 0.0;

    printf("{\"gpu\": \"%s\", \"sms\": %d, \"threads_per_sm\": %d, \"rates_per_clk_per_sm\": {", prop.name, g_sms,
           kThreads);
    auto report = [&](const char* name, double cycles, double scale, bool last = false) {
        printf("\"%s\": %.2f%s", name, lanes * scale / cycles, last ? "" : ", ");
    };
    report("ex2.approx.f32", run([&] { k_alu<0><<<grid, block>>>(0.3f, g_out, g_sink); }, &mhz), 1.0);
    report("lg2.approx.f32", run([&] { k_alu<1><<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr), 1.0);
    report("rcp.approx.f32", run([&] { k_alu<2><<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr), 1.0);
    report("tanh.approx.f32", run([&] { k_alu<3><<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr), 1.0);
    report("fma.f32 lanes", run([&] { k_alu<4><<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr), 1.0);
    report("fma.f32x2 lanes", run([&] { k_fma2<<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr), 2.0);
    report("mix: ex2 + 2 fma.f32x2 (ex2 count)", run([&] { k_mix<<<grid, block>>>(0.3f, g_out, g_sink); }, nullptr),
           1.0);
    // shared memory: bytes delivered to registers per clock
    report("lds.128 same address, bytes", run([&] { k_lds<0><<<grid, block>>>(g_out, g_sink); }, nullptr), 16.0);
    report("lds.128 two addresses, bytes", run([&] { k_lds<1><<<grid, block>>>(g_out, g_sink); }, nullptr), 16.0);
    report("lds.128 distinct, bytes", run([&] { k_lds<2><<<grid, block>>>(g_out, g_sink); }, nullptr), 16.0);
    report("lds.64 two addresses, bytes", run([&] { k_lds<4><<<grid, block>>>(g_out, g_sink); }, nullptr), 8.0);
    report("lds.32 same address, bytes", run([&] { k_lds<3><<<grid, block>>>(g_out, g_sink); }, nullptr), 4.0);
    report("shfl.idx lanes", run([&] { k_shfl<<<grid, block>>>(g_out, g_sink); }, nullptr), 1.0);
    // mma: multiply-adds per clock per SM (a warp instruction is 1/32 of the lane count)
    report("mma.sync m16n8k8 tf32 MACs", run([&] { k_mma<0><<<grid, block>>>(g_out, g_sink); }, nullptr),
           16.0 * 8 * 8 / 32.0);
    report("mma.sync m16n8k16 bf16 MACs", run([&] { k_mma<1><<<grid, block>>>(g_out, g_sink); }, nullptr),
           16.0 * 8 * 16 / 32.0, true);
    printf("}, \"state_update_loop_updates_per_clk_per_sm\": {");
    const int steps = 4096;
    const int warps_per_sm[] = {4, 8, 16};
    for (int wi = 0; wi < 3; ++wi) {
        const int thr = 32 * warps_per_sm[wi];
        const double upd = (double)thr * steps * 8;
        const double cp = run([&] { k_update<true, 8><<<grid, thr>>>(0.3f, g_out, g_sink, steps); }, nullptr);
        const double cs = run([&] { k_update<false, 8><<<grid, thr>>>(0.3f, g_out, g_sink, steps); }, nullptr);
        printf("\"%d warps, 8 states, packed\": %.2f, \"%d warps, 8 states, scalar\": %.2f%s", warps_per_sm[wi],
               upd / cp, warps_per_sm[wi], upd / cs, wi < 2 ? ", " : "");
    }
    printf("}, \"sm_mhz_during_ex2_run\": %.0f, \"method\": \"one 512-thread CTA per SM, %d x %d independent "
           "instances per thread, clock64 around the run; update loops: one CTA per SM of the given warps\"}\n",
           mhz, kIters, kUnroll);
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        fprintf(stderr, "CUDA error: %s\n", cudaGetErrorString(e));
        return 1;
    }
    return 0;
}
