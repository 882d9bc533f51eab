// Fast selective-scan kernels for dense channel-contiguous layouts (the Mamba block's
// (b, L, D) activations and (b, L, N) B, C), N in {16, 32, 64}, forward direction,
// delta*B discretisation; with an optional split of the sequence into chunks.
//
// Work split. A CTA owns kCh = 16 consecutive channels of one batch row and walks one
// chunk of the sequence (the whole sequence when it is not split). LPC lanes share a
// channel, lane g keeping the fp32 states n in [g S, g S + S), S = N / LPC, in registers.
//
// Data movement. TMA (3-D tensor maps over (D or N, L, b)) streams 32-step tiles of x,
// delta, z, B and C into a 3-deep shared-memory ring guarded by mbarriers; y tiles leave
// through TMA stores from a double buffer. B and C tiles are widened to fp32 once per tile
// by the CTA, so lanes then read their states' values with 8- or 16-byte loads.
//
// Steps go in groups of LPC. Lane g of a channel computes the per-(t, channel) scalars of
// step g of the group (dt = softplus(delta + bias), dt x, silu(z), D x) one group ahead, so
// that chain overlaps the state updates of the current group; the (dt, dt x) pairs are then
// broadcast inside the channel's lanes. Per step and state:
//   A_bar[n] = 2^(dt * A[n] * log2 e)           SFU ex2
//   h[n] = A_bar[n] h[n] + (dt x) B[n]          packed fp32 pairs (fma.rn.f32x2)
//   y += C[n] h[n]                               packed pairs
// and the lanes' partial sums of the LPC steps are reduce-scattered (log2 LPC shuffle
// rounds), leaving lane g with step g's y, which it finishes as (y + D x) silu(z).
//
// Chunked sequence (long sequences with few channels, where one CTA per channel tile
// would leave most SMs idle):
//  * pass 1 (kPass1): every chunk but the last runs from a zero state without the readout
//    and writes its local end state and the sum of its dt (per channel) to the workspace;
//  * carry kernel: per (b, d, n), H_0 = h0, H_{c+1} = exp(A sum_dt_c) H_c + local_c, in
//    chunk order, written back in place as the initial state of chunk c + 1;
//  * pass 2 (kFull): every chunk runs from its initial state and writes y; the last chunk
//    also writes h_last.
// The split uses the associativity of the recurrence h -> A_bar h + b: a chunk's map is
// h -> (prod A_bar) h + (its zero-start end state), and prod A_bar = exp(A sum dt).
//
// Recurrence: "Mamba/SSM complete guide" section 5 `selective_scan` and MambaBlock.forward;
// "論文解説: Mamba" "選択機構" (softplus) and "Hardware-Aware Parallel Scan" (state kept
// on chip, only the outputs written back; the parallel scan over (A_bar, B_bar x) pairs).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kCh = 16;        // channels per CTA
constexpr int kT = 32;         // steps per tile
constexpr int kStages = 3;     // TMA ring depth

enum Mode { kFull = 0, kPass1 = 1 };

struct FastParams {
    int64_t seqlen;
    int64_t chunk;         // steps per chunk (multiple of kT); >= seqlen when not split
    int dim;
    int nchunks;
    const float* A;
    const float* D;
    const float* bias;
    const float* h0;
    float* h_last;
    float* carry;          // (nchunks - 1, b, D, N): local end states, then initial states
    float* sumdt;          // (nchunks - 1, b, D)
    unsigned* status;
    int skip_first_load;   // test hook: never issue tile 0 (only used when the sequence is one tile)
};

template <int N, bool BF16>
struct Layout {
    static constexpr int kEsz = BF16 ? 2 : 4;
    static constexpr int kTileX = kT * kCh * kEsz;          // one of x, delta, z, y
    static constexpr int kTileB = kT * N * kEsz;            // one of B, C
    static constexpr int kStageBytes = 3 * kTileX + 2 * kTileB;
    static constexpr int kStageStride = (kStageBytes + 127) / 128 * 128;
    static constexpr int kBars = 0;                                   // kStages mbarriers
    static constexpr int kRing = 128;
    static constexpr int kBCf = kRing + kStages * kStageStride;       // fp32 B then C [kT][N]
    static constexpr int kY = kBCf + 2 * kT * N * 4;                  // 2 y tiles
    static constexpr int kYStride = (kTileX + 127) / 128 * 128;
    static constexpr int kTotal = kY + 2 * kYStride;
};

__device__ __forceinline__ float ld_io(const void* base, int i, bool bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]) : static_cast<const float*>(base)[i];
}

// Per-(step, channel) scalars one lane computes for its step of a group.
struct Scal {
    float dt, u, dx, gate;
};

template <bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS>
__device__ __forceinline__ Scal scalars(const void* xs, const void* ds, const void* zs, int jj, int c, float bias,
                                        float Dd, bool tv) {
    Scal r;
    const float xr = ld_io(xs, jj * kCh + c, BF16);
    float dt = ld_io(ds, jj * kCh + c, BF16) + bias;
    if constexpr (SOFTPLUS) dt = softplus_fast(dt);
    r.dt = tv ? dt : 0.f;
    r.u = r.dt * xr;
    r.dx = DSKIP ? Dd * xr : 0.f;
    r.gate = GATE ? silu_fast(ld_io(zs, jj * kCh + c, BF16)) : 1.f;
    return r;
}

// S consecutive fp32 values of a shared-memory row as S / 2 packed pairs.
template <int S>
__device__ __forceinline__ void lds_pairs(const float* p, f2 (&v)[S / 2]) {
    if constexpr (S % 4 == 0) {
#pragma unroll
        for (int k = 0; k < S / 2; k += 2) {
            const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(p + 2 * k);
            v[k] = q.x;
            v[k + 1] = q.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < S / 2; ++k) v[k] = *reinterpret_cast<const unsigned long long*>(p + 2 * k);
    }
}

template <int N, bool BF16, int LPC, bool GATE, bool DSKIP, bool SOFTPLUS, int MODE>
__global__ void __launch_bounds__(kCh * LPC, 16 / LPC)
scan_fast_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap md,
                 const __grid_constant__ CUtensorMap mz, const __grid_constant__ CUtensorMap mB,
                 const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap my,
                 const FastParams p) {
    using Lay = Layout<N, BF16>;
    constexpr int kThreads = kCh * LPC;
    constexpr int S = N / LPC;         // states per lane
    constexpr int P = S / 2;           // packed pairs per lane
    constexpr bool kReadout = MODE == kFull;
    constexpr bool kGate = GATE && kReadout;
    static_assert(S % 2 == 0, "states per lane must be even");
    static_assert(LPC == 2 || LPC == 4 || LPC == 8, "2, 4 or 8 lanes per channel");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBars);

    const int tid = threadIdx.x;
    const int c = tid / LPC, g = tid % LPC;
    const int d0 = blockIdx.x * kCh;
    const int b = blockIdx.y;
    const int chunk = blockIdx.z;
    const int d = d0 + c;
    const bool dvalid = d < p.dim;
    const int64_t t_begin = (int64_t)chunk * p.chunk;
    const int64_t t_end = t_begin + p.chunk < p.seqlen ? t_begin + p.chunk : p.seqlen;
    const int64_t len = t_end - t_begin;
    const int ntiles = (int)((len + kT - 1) / kT);

    // initial state: h0 for the first chunk, the carried state for the others (pass 2),
    // zero in pass 1
    const float* hinit = nullptr;
    if constexpr (MODE == kFull) {
        if (chunk == 0)
            hinit = p.h0 ? p.h0 + ((int64_t)b * p.dim) * N : nullptr;
        else
            hinit = p.carry + ((int64_t)(chunk - 1) * gridDim.y + b) * p.dim * N;
    }
    f2 A2[P], h[P];
#pragma unroll
    for (int k = 0; k < P; ++k) {
        const int n = g * S + 2 * k;
        float a0 = 0.f, a1 = 0.f, h0v = 0.f, h1v = 0.f;
        if (dvalid) {
            a0 = p.A[(int64_t)d * N + n] * kLog2e;
            a1 = p.A[(int64_t)d * N + n + 1] * kLog2e;
            if (hinit) {
                h0v = hinit[(int64_t)d * N + n];
                h1v = hinit[(int64_t)d * N + n + 1];
            }
        }
        A2[k] = pk(a0, a1);
        h[k] = pk(h0v, h1v);
    }
    const float bias = (dvalid && p.bias) ? p.bias[d] : 0.f;
    const float Dd = (DSKIP && dvalid) ? p.D[d] : 0.f;
    float dtsum = 0.f;   // pass 1: sum of dt over the chunk

    auto stage_ptr = [&](int buf) { return smem + Lay::kRing + buf * Lay::kStageStride; };
    auto issue = [&](int s) {
        const int buf = s % kStages;
        unsigned char* st = stage_ptr(buf);
        constexpr unsigned kBytes = Lay::kStageBytes - (kGate ? 0 : Lay::kTileX) - (kReadout ? 0 : Lay::kTileB);
        mbar_arrive_expect_tx(&bars[buf], kBytes);
        const int t0 = (int)(t_begin + (int64_t)s * kT);
        tma_load_3d(st, &mx, d0, t0, b, &bars[buf]);
        tma_load_3d(st + Lay::kTileX, &md, d0, t0, b, &bars[buf]);
        if constexpr (kGate) tma_load_3d(st + 2 * Lay::kTileX, &mz, d0, t0, b, &bars[buf]);
        tma_load_3d(st + 3 * Lay::kTileX, &mB, 0, t0, b, &bars[buf]);
        if constexpr (kReadout) tma_load_3d(st + 3 * Lay::kTileX + Lay::kTileB, &mC, 0, t0, b, &bars[buf]);
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&mx);
        prefetch_tensormap(&mB);
        for (int s = p.skip_first_load ? 1 : 0; s < kStages && s < ntiles; ++s) issue(s);
    }
    __syncthreads();

    bool failed = false;
    for (int s = 0; s < ntiles; ++s) {
        const int buf = s % kStages;
        const bool ok = mbar_wait_bounded(&bars[buf], (s / kStages) & 1, p.status);
        if (__syncthreads_or(!ok)) {
            // give up on this tile; before leaving, wait (bounded) for the later tiles
            // already issued so that no copy still targets this CTA's shared memory
            if (tid == 0)
                for (int s2 = s + 1; s2 < s + kStages && s2 < ntiles; ++s2)
                    mbar_wait_bounded(&bars[s2 % kStages], (s2 / kStages) & 1, p.status);
            failed = true;
            break;
        }
        unsigned char* st = stage_ptr(buf);
        const void* xs = st;
        const void* ds = st + Lay::kTileX;
        const void* zs = st + 2 * Lay::kTileX;
        // B (and C) of the tile widened to fp32
        float* bcf = reinterpret_cast<float*>(smem + Lay::kBCf);
        if constexpr (BF16) {
            const uint4* src = reinterpret_cast<const uint4*>(st + 3 * Lay::kTileX);
            constexpr int kChunks = (kReadout ? 2 : 1) * kT * N / 8;
#pragma unroll
            for (int i = tid; i < kChunks; i += kThreads) {
                const uint4 v = src[i];
                float4* dst = reinterpret_cast<float4*>(bcf + i * 8);
                dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                     __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(st + 3 * Lay::kTileX);
            constexpr int kChunks = (kReadout ? 2 : 1) * kT * N / 4;
#pragma unroll
            for (int i = tid; i < kChunks; i += kThreads) reinterpret_cast<float4*>(bcf)[i] = src[i];
        }
        const float* Bf = bcf;
        const float* Cf = bcf + kT * N;
        unsigned char* ys = smem + Lay::kY + (s & 1) * Lay::kYStride;
        if (kReadout && s >= 2 && tid == 0) tma_store_wait_read<1>();   // the store of tile s-2 read ys
        __syncthreads();
        const int rem = (int)(len - (int64_t)s * kT);
        const int tcount = rem < kT ? rem : kT;

        float yout[kT / LPC];   // the steps this lane finishes; stored after the loop so that no
                                // shared-memory store sits between the loads of later steps
        Scal cur = scalars<BF16, kGate, DSKIP && kReadout, SOFTPLUS>(xs, ds, zs, g, c, bias, Dd, g < tcount);
#pragma unroll
        for (int grp = 0; grp < kT / LPC; ++grp) {
            // the next group's scalars: independent of the state, overlaps the updates below
            const int jn = (grp + 1) * LPC + g;
            const Scal nxt = scalars<BF16, kGate, DSKIP && kReadout, SOFTPLUS>(xs, ds, zs, jn < kT ? jn : g, c, bias,
                                                                              Dd, jn < tcount);
            float acc[LPC];
#pragma unroll
            for (int q = 0; q < LPC; ++q) {
                const float dtq = __shfl_sync(0xffffffffu, cur.dt, q, LPC);
                const float uq = __shfl_sync(0xffffffffu, cur.u, q, LPC);
                if constexpr (MODE == kPass1) dtsum += dtq;
                const f2 dt2 = pk(dtq, dtq), u2 = pk(uq, uq);
                f2 bv[P];
                lds_pairs<S>(Bf + (grp * LPC + q) * N + g * S, bv);
                f2 cv[P];
                if constexpr (kReadout) lds_pairs<S>(Cf + (grp * LPC + q) * N + g * S, cv);
                f2 a2 = pk(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    float e0, e1;
                    upk(mul2(dt2, A2[k]), e0, e1);
                    const f2 ab = pk(ex2_approx(e0), ex2_approx(e1));
                    h[k] = fma2(ab, h[k], mul2(u2, bv[k]));
                    if constexpr (kReadout) a2 = fma2(cv[k], h[k], a2);
                }
                if constexpr (kReadout) {
                    float lo, hi;
                    upk(a2, lo, hi);
                    acc[q] = lo + hi;
                }
            }
            if constexpr (kReadout) {
                // reduce-scatter over the LPC lanes of the channel: each round a lane keeps the
                // half of its partial sums whose step index has its lane bit and adds the
                // partner's; lane g ends with the full sum of step g
#pragma unroll
                for (int m = LPC / 2; m >= 1; m >>= 1) {
                    const bool upper = (g & m) != 0;
#pragma unroll
                    for (int i = 0; i < m; ++i) {
                        const float keep = upper ? acc[i + m] : acc[i];
                        const float send = upper ? acc[i] : acc[i + m];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
                yout[grp] = (acc[0] + cur.dx) * cur.gate;
            }
            cur = nxt;
        }
        if constexpr (kReadout) {
#pragma unroll
            for (int grp = 0; grp < kT / LPC; ++grp) {
                const int jj = grp * LPC + g;
                if constexpr (BF16)
                    reinterpret_cast<__nv_bfloat16*>(ys)[jj * kCh + c] = __float2bfloat16_rn(yout[grp]);
                else
                    reinterpret_cast<float*>(ys)[jj * kCh + c] = yout[grp];
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            if constexpr (kReadout) {
                tma_store_3d(&my, d0, (int)(t_begin + (int64_t)s * kT), b, ys);
                tma_store_commit();
            }
            if (s + kStages < ntiles) issue(s + kStages);
        }
    }
    if (kReadout && tid == 0) tma_store_wait_all();
    if (failed) return;
    if (!dvalid) return;
    if constexpr (MODE == kFull) {
        if (p.h_last && chunk == (int)gridDim.z - 1) {
            float* out = p.h_last + ((int64_t)b * p.dim + d) * N;
#pragma unroll
            for (int k = 0; k < P; ++k) {
                float lo, hi;
                upk(h[k], lo, hi);
                *reinterpret_cast<float2*>(out + g * S + 2 * k) = make_float2(lo, hi);
            }
        }
    } else {
        float* out = p.carry + (((int64_t)chunk * gridDim.y + b) * p.dim + d) * N;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            float lo, hi;
            upk(h[k], lo, hi);
            *reinterpret_cast<float2*>(out + g * S + 2 * k) = make_float2(lo, hi);
        }
        if (g == 0) p.sumdt[((int64_t)chunk * gridDim.y + b) * p.dim + d] = dtsum;
    }
}

// Chunk carry: one thread per (b, d, n) walks the chunks in order,
//   H_0 = h0,  H_{c+1} = exp(A[d, n] * sumdt_c) * H_c + local_c,
// and stores H_{c+1} over local_c (the initial state of chunk c + 1).
__global__ void scan_carry_kernel(float* carry, const float* sumdt, const float* A, const float* h0,
                                  int64_t batch, int64_t dim, int N, int nsteps) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = batch * dim * N;
    if (i >= total) return;
    const int64_t bd = i / N;
    const int n = (int)(i % N);
    const int64_t d = bd % dim;
    const float a = A[d * N + n];
    float H = h0 ? h0[i] : 0.f;
    for (int c = 0; c < nsteps; ++c) {
        const int64_t o = (int64_t)c * total + i;
        H = fmaf(expf(a * sumdt[(int64_t)c * batch * dim + bd]), H, carry[o]);
        carry[o] = H;
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D map over (inner, L, b) with element strides (1, st, sb) and box (box0, kT, 1).
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t L, int64_t b, int64_t st,
              int64_t sb, int box0) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)b};
    const int64_t bstride = b > 1 ? sb * esz : ((L * st * esz + 15) / 16) * 16;
    cuuint64_t strides[2] = {(cuuint64_t)(st * esz), (cuuint64_t)bstride};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)kT, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                    const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Lanes per channel: N / 8, so every lane keeps 8 states (4 packed pairs). Measured on the
// b8 D1536 L2048 N16 bf16 workload: 2 lanes 177 us, 4 lanes 194 us, 8 lanes 236 us -- eight
// independent state chains per lane hide the SFU and shared-memory latency better than more
// warps with fewer states each.
template <int N>
constexpr int lanes_per_channel() { return N / 8; }

template <int N, bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS, int MODE, int LPC = lanes_per_channel<N>()>
cudaError_t launch_t(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz, cudaStream_t st) {
    using Lay = Layout<N, BF16>;
    auto kern = scan_fast_kernel<N, BF16, LPC, GATE, DSKIP, SOFTPLUS, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kTotal);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + kCh - 1) / kCh), (unsigned)a.batch, (unsigned)nz);
    kern<<<grid, kCh * LPC, Lay::kTotal, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], fp);
    note_launches(1);
    return cudaGetLastError();
}

template <int N, bool BF16, int MODE>
cudaError_t dispatch_flags(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz, cudaStream_t st) {
    const bool gate = a.z != nullptr, dskip = a.D != nullptr, sp = a.softplus != 0;
    if constexpr (MODE == kPass1) {
        // pass 1 reads neither z nor D
        return sp ? launch_t<N, BF16, false, false, true, MODE>(maps, fp, a, nz, st)
                  : launch_t<N, BF16, false, false, false, MODE>(maps, fp, a, nz, st);
    } else {
#define SSM_FAST_CASE(G_, D_, S_) \
    if (gate == G_ && dskip == D_ && sp == S_) return launch_t<N, BF16, G_, D_, S_, MODE>(maps, fp, a, nz, st);
        SSM_FAST_CASE(true, true, true)
        SSM_FAST_CASE(true, true, false)
        SSM_FAST_CASE(true, false, true)
        SSM_FAST_CASE(true, false, false)
        SSM_FAST_CASE(false, true, true)
        SSM_FAST_CASE(false, true, false)
        SSM_FAST_CASE(false, false, true)
        SSM_FAST_CASE(false, false, false)
#undef SSM_FAST_CASE
    }
    return cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t dispatch(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz, cudaStream_t st) {
    const bool bf = a.io_bf16 != 0;
    switch (a.dstate) {
        case 16: return bf ? dispatch_flags<16, true, MODE>(maps, fp, a, nz, st)
                           : dispatch_flags<16, false, MODE>(maps, fp, a, nz, st);
        case 32: return bf ? dispatch_flags<32, true, MODE>(maps, fp, a, nz, st)
                           : dispatch_flags<32, false, MODE>(maps, fp, a, nz, st);
        case 64: return bf ? dispatch_flags<64, true, MODE>(maps, fp, a, nz, st)
                           : dispatch_flags<64, false, MODE>(maps, fp, a, nz, st);
    }
    return cudaErrorInvalidValue;
}

constexpr int64_t kMinChunk = 512;    // shortest chunk the automatic split uses

}  // namespace

bool scan_fast_supported(const ScanArgs& a) {
    const int N = a.dstate;
    if (N != 16 && N != 32 && N != 64) return false;
    if (a.reverse || a.zoh) return false;
    if (a.batch > 65535 || a.dim > (int64_t)1 << 30 || a.seqlen > ((int64_t)1 << 31) - 2 * kT) return false;
    if (!encode_fn()) return false;
    const int64_t esz = a.io_bf16 ? 2 : 4;
    auto act_ok = [&](const void* ptr, const int64_t* s) {
        if (!ptr) return true;
        if (!aligned16(ptr) || s[2] != 1) return false;
        if ((s[1] * esz) % 16 || s[1] < a.dim) return false;
        if (a.batch > 1 && ((s[0] * esz) % 16 || s[0] == 0)) return false;
        return true;
    };
    auto bc_ok = [&](const void* ptr, const int64_t* s) {
        if (!aligned16(ptr) || s[2] != 1) return false;
        if ((s[1] * esz) % 16 || s[1] < N || (N * esz) % 16) return false;
        if (a.batch > 1 && ((s[0] * esz) % 16 || s[0] == 0)) return false;
        return true;
    };
    return act_ok(a.x, a.xs) && act_ok(a.delta, a.ds) && act_ok(a.z, a.zs) && act_ok(a.y, a.ys) &&
           bc_ok(a.B, a.Bs) && bc_ok(a.C, a.Cs);
}

int64_t scan_fast_chunk(const ScanArgs& a) {
    const int64_t L = a.seqlen;
    int64_t q;
    if (a.chunk_len > 0) {
        q = a.chunk_len;
    } else {
        // split only when the channel tiles leave the SMs short of work
        const int64_t tiles = a.batch * ((a.dim + kCh - 1) / kCh);
        const int64_t want = 8 * 148;
        if (tiles >= 2 * 148 || L < 2 * kMinChunk) return ((L + kT - 1) / kT) * kT;
        int64_t nch = (want + tiles - 1) / tiles;
        q = (L + nch - 1) / nch;
        if (q < kMinChunk) q = kMinChunk;
    }
    q = ((q + kT - 1) / kT) * kT;
    if (q >= L) q = ((L + kT - 1) / kT) * kT;
    return q;
}

size_t scan_fast_workspace_bytes(const ScanArgs& a) {
    if (a.seqlen == 0) return 0;
    const int64_t q = scan_fast_chunk(a);
    const int64_t nch = (a.seqlen + q - 1) / q;
    if (nch <= 1) return 0;
    return (size_t)((nch - 1) * a.batch * a.dim * (a.dstate + 1)) * sizeof(float);
}

cudaError_t launch_scan_fast(const ScanArgs& a, cudaStream_t st) {
    CUtensorMap maps[6];
    const bool bf = a.io_bf16 != 0;
    const void* zsrc = a.z ? a.z : a.x;                 // unused map when there is no gate
    const int64_t* zst = a.z ? a.zs : a.xs;
    if (!make_map(&maps[0], a.x, bf, a.dim, a.seqlen, a.batch, a.xs[1], a.xs[0], kCh) ||
        !make_map(&maps[1], a.delta, bf, a.dim, a.seqlen, a.batch, a.ds[1], a.ds[0], kCh) ||
        !make_map(&maps[2], zsrc, bf, a.dim, a.seqlen, a.batch, zst[1], zst[0], kCh) ||
        !make_map(&maps[3], a.B, bf, a.dstate, a.seqlen, a.batch, a.Bs[1], a.Bs[0], a.dstate) ||
        !make_map(&maps[4], a.C, bf, a.dstate, a.seqlen, a.batch, a.Cs[1], a.Cs[0], a.dstate) ||
        !make_map(&maps[5], a.y, bf, a.dim, a.seqlen, a.batch, a.ys[1], a.ys[0], kCh))
        return cudaErrorInvalidValue;
    const int64_t q = scan_fast_chunk(a);
    const int nch = (int)((a.seqlen + q - 1) / q);
    FastParams fp{a.seqlen, q, (int)a.dim, nch, a.A, a.D, a.bias, a.h0, a.h_last, nullptr, nullptr,
                  device_status_ptr(), (a.debug_flags & SSM_DEBUG_SKIP_FIRST_LOAD) ? 1 : 0};
    if (!fp.status) return cudaErrorInvalidValue;
    if (nch > 1) {
        const size_t carry_floats = (size_t)((nch - 1) * a.batch * a.dim * a.dstate);
        fp.carry = static_cast<float*>(a.workspace);
        fp.sumdt = fp.carry + carry_floats;
        cudaError_t e = dispatch<kPass1>(maps, fp, a, nch - 1, st);
        if (e != cudaSuccess) return e;
        const int64_t total = a.batch * a.dim * a.dstate;
        scan_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(fp.carry, fp.sumdt, a.A, a.h0, a.batch,
                                                                          a.dim, a.dstate, nch - 1);
        note_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return dispatch<kFull>(maps, fp, a, nch, st);
}

}  // namespace ssm
