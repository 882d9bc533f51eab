// Fast selective-scan kernel for dense channel-contiguous layouts (the Mamba block's
// (b, L, D) activations and (b, L, N) B, C), N in {16, 32, 64}, forward direction,
// delta*B discretisation.
//
// Work split. A CTA is two warps and owns 16 consecutive channels of one batch row for the
// whole sequence; four lanes 4c..4c+3 share channel c, each holding N/4 fp32 states in
// registers (config b8 D1536 N16: 1536 warps, ~10 per SM, 4 states per lane).
//
// Data movement. TMA (3-D tensor maps over (D or N, L, b)) streams 32-step tiles of x,
// delta, z, B and C into a 3-deep shared-memory ring guarded by mbarriers; y tiles leave
// through TMA stores from a double buffer. B and C tiles are widened to fp32 once per stage
// by the CTA, so every lane then reads its N/4 values with 16-byte loads.
//
// Steps go in groups of four. Lane g of a channel computes the per-(t, channel) scalars of
// step g of the group (softplus(delta + bias), dt x, silu(z)) one group ahead, so that
// chain overlaps the state updates of the current group; the four (dt, dt x) pairs are then
// broadcast inside the channel's lanes. Per step and state:
//   A_bar[n] = 2^(dt * A[n] * log2 e)           SFU ex2
//   h[n] = A_bar[n] h[n] + (dt x) B[n]          packed fp32 pairs (fma.rn.f32x2)
//   y += C[n] h[n]                               packed pairs
// and the four lanes' partial sums of the four steps are reduce-scattered (two shuffle
// rounds), leaving lane g with step g's y, which it finishes as (y + D x) silu(z).
//
// Recurrence: "Mamba/SSM complete guide" section 5 `selective_scan` and MambaBlock.forward;
// "論文解説: Mamba" "選択機構" (softplus) and "Hardware-Aware Parallel Scan" (state kept
// on chip, only the outputs written back).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kCh = 16;        // channels per CTA
constexpr int kG = 4;          // lanes per channel
constexpr int kThreads = kCh * kG;
constexpr int kT = 32;         // steps per stage
constexpr int kStages = 3;     // TMA ring depth

struct FastParams {
    int64_t seqlen;
    int dim;
    const float* A;
    const float* D;
    const float* bias;
    const float* h0;
    float* h_last;
    unsigned* status;
    int skip_first_load;   // test hook: never issue stage 0 (only used when the sequence is one stage)
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
    static constexpr int kBCf = kRing + kStages * kStageStride;       // fp32 B, C (bf16 I/O)
    static constexpr int kBCfBytes = BF16 ? 2 * kT * N * 4 : 0;
    static constexpr int kY = kBCf + (kBCfBytes + 127) / 128 * 128;   // 2 y tiles
    static constexpr int kYStride = (kTileX + 127) / 128 * 128;
    static constexpr int kTotal = kY + 2 * kYStride;
};

__device__ __forceinline__ float ld_io(const void* base, int i, bool bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]) : static_cast<const float*>(base)[i];
}

// Sixteen bytes of shared memory as two packed fp32 pairs.
__device__ __forceinline__ void lds_2xf2(const float* p, f2& lo, f2& hi) {
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
    lo = v.x;
    hi = v.y;
}

// Per-(step, channel) scalars one lane computes for its step of a group.
struct Scal {
    float dt, u, xr, gate;
};

template <bool BF16, bool GATE, bool SOFTPLUS>
__device__ __forceinline__ Scal scalars(const void* xs, const void* ds, const void* zs, int jj, int c, float bias,
                                        bool tv) {
    Scal r;
    r.xr = ld_io(xs, jj * kCh + c, BF16);
    float dt = ld_io(ds, jj * kCh + c, BF16) + bias;
    if constexpr (SOFTPLUS) dt = softplus_fast(dt);
    r.dt = tv ? dt : 0.f;
    r.u = r.dt * r.xr;
    r.gate = GATE ? silu_fast(ld_io(zs, jj * kCh + c, BF16)) : 1.f;
    return r;
}

template <int N, bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS>
__global__ void __launch_bounds__(kThreads)
scan_fast_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap md,
                 const __grid_constant__ CUtensorMap mz, const __grid_constant__ CUtensorMap mB,
                 const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap my,
                 const FastParams p) {
    using Lay = Layout<N, BF16>;
    constexpr int S = N / kG;          // states per lane
    constexpr int P = S / 2;           // packed pairs per lane
    static_assert(S % 4 == 0, "states per lane must be a multiple of 4");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBars);

    const int tid = threadIdx.x;
    const int c = tid / kG, g = tid % kG;
    const int d0 = blockIdx.x * kCh;
    const int b = blockIdx.y;
    const int d = d0 + c;
    const bool dvalid = d < p.dim;
    const int64_t L = p.seqlen;
    const int nst = (int)((L + kT - 1) / kT);

    f2 A2[P], h[P];
#pragma unroll
    for (int k = 0; k < P; ++k) {
        const int n = g * S + 2 * k;
        float a0 = 0.f, a1 = 0.f, h0v = 0.f, h1v = 0.f;
        if (dvalid) {
            a0 = p.A[(int64_t)d * N + n] * kLog2e;
            a1 = p.A[(int64_t)d * N + n + 1] * kLog2e;
            if (p.h0) {
                h0v = p.h0[((int64_t)b * p.dim + d) * N + n];
                h1v = p.h0[((int64_t)b * p.dim + d) * N + n + 1];
            }
        }
        A2[k] = pk(a0, a1);
        h[k] = pk(h0v, h1v);
    }
    const float bias = (dvalid && p.bias) ? p.bias[d] : 0.f;
    const float Dd = (DSKIP && dvalid) ? p.D[d] : 0.f;

    auto stage_ptr = [&](int buf) { return smem + Lay::kRing + buf * Lay::kStageStride; };
    auto issue = [&](int s) {
        const int buf = s % kStages;
        unsigned char* st = stage_ptr(buf);
        mbar_arrive_expect_tx(&bars[buf], Lay::kStageBytes - (GATE ? 0 : Lay::kTileX));
        const int t0 = s * kT;
        tma_load_3d(st, &mx, d0, t0, b, &bars[buf]);
        tma_load_3d(st + Lay::kTileX, &md, d0, t0, b, &bars[buf]);
        if constexpr (GATE) tma_load_3d(st + 2 * Lay::kTileX, &mz, d0, t0, b, &bars[buf]);
        tma_load_3d(st + 3 * Lay::kTileX, &mB, 0, t0, b, &bars[buf]);
        tma_load_3d(st + 3 * Lay::kTileX + Lay::kTileB, &mC, 0, t0, b, &bars[buf]);
    };

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&mx);
        prefetch_tensormap(&mB);
        for (int s = p.skip_first_load ? 1 : 0; s < kStages && s < nst; ++s) issue(s);
    }
    __syncthreads();

    bool failed = false;
    for (int s = 0; s < nst; ++s) {
        const int buf = s % kStages;
        const bool ok = mbar_wait_bounded(&bars[buf], (s / kStages) & 1, p.status);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        unsigned char* st = stage_ptr(buf);
        const void* xs = st;
        const void* ds = st + Lay::kTileX;
        const void* zs = st + 2 * Lay::kTileX;
        const float* Bf;
        const float* Cf;
        if constexpr (BF16) {
            float* bcf = reinterpret_cast<float*>(smem + Lay::kBCf);
            const uint4* src = reinterpret_cast<const uint4*>(st + 3 * Lay::kTileX);   // B then C, bf16
            constexpr int kChunks = 2 * kT * N / 8;
#pragma unroll
            for (int i = tid; i < kChunks; i += kThreads) {
                const uint4 v = src[i];
                float4* dst = reinterpret_cast<float4*>(bcf + i * 8);
                dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                     __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            }
            Bf = bcf;
            Cf = bcf + kT * N;
        } else {
            Bf = reinterpret_cast<const float*>(st + 3 * Lay::kTileX);
            Cf = reinterpret_cast<const float*>(st + 3 * Lay::kTileX + Lay::kTileB);
        }
        unsigned char* ys = smem + Lay::kY + (s & 1) * Lay::kYStride;
        if (s >= 2 && tid == 0) tma_store_wait_read<1>();
        __syncthreads();
        const int64_t rem = L - (int64_t)s * kT;
        const int tcount = rem < kT ? (int)rem : kT;
        const int ngrp = (tcount + kG - 1) / kG;

        Scal cur = scalars<BF16, GATE, SOFTPLUS>(xs, ds, zs, g, c, bias, g < tcount);
#pragma unroll 2
        for (int grp = 0; grp < kT / kG; ++grp) {
            if (grp >= ngrp) break;
            // the next group's scalars: independent of the state, overlaps the updates below
            const int jn = (grp + 1) * kG + g;
            Scal nxt = scalars<BF16, GATE, SOFTPLUS>(xs, ds, zs, jn < kT ? jn : g, c, bias, jn < tcount);

            float acc[kG];
#pragma unroll
            for (int q = 0; q < kG; ++q) {
                const float dtq = __shfl_sync(0xffffffffu, cur.dt, q, kG);
                const float uq = __shfl_sync(0xffffffffu, cur.u, q, kG);
                const f2 dt2 = pk(dtq, dtq), u2 = pk(uq, uq);
                const float* Brow = Bf + (grp * kG + q) * N + g * S;
                const float* Crow = Cf + (grp * kG + q) * N + g * S;
                f2 a2 = pk(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < P; k += 2) {
                    f2 b01, b23, c01, c23;
                    lds_2xf2(Brow + 2 * k, b01, b23);
                    lds_2xf2(Crow + 2 * k, c01, c23);
                    float e0, e1, e2, e3;
                    upk(mul2(dt2, A2[k]), e0, e1);
                    upk(mul2(dt2, A2[k + 1]), e2, e3);
                    const f2 ab01 = pk(ex2_approx(e0), ex2_approx(e1));
                    const f2 ab23 = pk(ex2_approx(e2), ex2_approx(e3));
                    h[k] = fma2(ab01, h[k], mul2(u2, b01));
                    h[k + 1] = fma2(ab23, h[k + 1], mul2(u2, b23));
                    a2 = fma2(c01, h[k], a2);
                    a2 = fma2(c23, h[k + 1], a2);
                }
                float lo, hi;
                upk(a2, lo, hi);
                acc[q] = lo + hi;
            }
            // reduce-scatter: lane g ends with the full sum of step g
            const bool hi2 = (g & 2) != 0;
            const float ra = (hi2 ? acc[2] : acc[0]) + __shfl_xor_sync(0xffffffffu, hi2 ? acc[0] : acc[2], 2);
            const float rb = (hi2 ? acc[3] : acc[1]) + __shfl_xor_sync(0xffffffffu, hi2 ? acc[1] : acc[3], 2);
            const bool hi1 = (g & 1) != 0;
            const float tot = (hi1 ? rb : ra) + __shfl_xor_sync(0xffffffffu, hi1 ? ra : rb, 1);
            const int jj = grp * kG + g;
            if (jj < tcount) {
                float out = DSKIP ? fmaf(Dd, cur.xr, tot) : tot;
                if constexpr (GATE) out *= cur.gate;
                if constexpr (BF16)
                    reinterpret_cast<__nv_bfloat16*>(ys)[jj * kCh + c] = __float2bfloat16_rn(out);
                else
                    reinterpret_cast<float*>(ys)[jj * kCh + c] = out;
            }
            cur = nxt;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&my, d0, s * kT, b, ys);
            tma_store_commit();
            if (s + kStages < nst) issue(s + kStages);
        }
    }
    if (tid == 0) tma_store_wait_all();
    if (failed) return;
    if (dvalid && p.h_last) {
#pragma unroll
        for (int k = 0; k < P; ++k) {
            float lo, hi;
            upk(h[k], lo, hi);
            const int n = g * S + 2 * k;
            p.h_last[((int64_t)b * p.dim + d) * N + n] = lo;
            p.h_last[((int64_t)b * p.dim + d) * N + n + 1] = hi;
        }
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

template <int N, bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS>
cudaError_t launch_t(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, cudaStream_t st) {
    using Lay = Layout<N, BF16>;
    auto kern = scan_fast_kernel<N, BF16, GATE, DSKIP, SOFTPLUS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kTotal);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + kCh - 1) / kCh), (unsigned)a.batch);
    kern<<<grid, kThreads, Lay::kTotal, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], fp);
    note_launches(1);
    return cudaGetLastError();
}

template <int N, bool BF16>
cudaError_t dispatch_flags(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, cudaStream_t st) {
    const bool gate = a.z != nullptr, dskip = a.D != nullptr, sp = a.softplus != 0;
#define SSM_FAST_CASE(G_, D_, S_) \
    if (gate == G_ && dskip == D_ && sp == S_) return launch_t<N, BF16, G_, D_, S_>(maps, fp, a, st);
    SSM_FAST_CASE(true, true, true)
    SSM_FAST_CASE(true, true, false)
    SSM_FAST_CASE(true, false, true)
    SSM_FAST_CASE(true, false, false)
    SSM_FAST_CASE(false, true, true)
    SSM_FAST_CASE(false, true, false)
    SSM_FAST_CASE(false, false, true)
    SSM_FAST_CASE(false, false, false)
#undef SSM_FAST_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool scan_fast_supported(const ScanArgs& a) {
    const int N = a.dstate;
    if (N != 16 && N != 32 && N != 64) return false;
    if (a.reverse || a.zoh) return false;
    if (a.batch > 65535 || a.dim > (int64_t)1 << 30 || a.seqlen > ((int64_t)1 << 31) - kT) return false;
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
    FastParams fp{a.seqlen, (int)a.dim, a.A, a.D, a.bias, a.h0, a.h_last, device_status_ptr(),
                  (a.debug_flags & SSM_DEBUG_SKIP_FIRST_LOAD) ? 1 : 0};
    if (!fp.status) return cudaErrorInvalidValue;
    switch (a.dstate) {
        case 16: return bf ? dispatch_flags<16, true>(maps, fp, a, st) : dispatch_flags<16, false>(maps, fp, a, st);
        case 32: return bf ? dispatch_flags<32, true>(maps, fp, a, st) : dispatch_flags<32, false>(maps, fp, a, st);
        case 64: return bf ? dispatch_flags<64, true>(maps, fp, a, st) : dispatch_flags<64, false>(maps, fp, a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssm
