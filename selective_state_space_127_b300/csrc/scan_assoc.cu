// Selective scan with an in-tile associative scan over (A_bar, B_bar x) pairs: the form the
// pages give for the parallel scan, offered as an alternative algorithm of ssm_scan_fwd
// (SSM_SCAN_ALGO_ASSOC) beside the default serial walk of scan_fast.cuh.
//
// Work split. A CTA of 16 warps owns kCh = 16 consecutive channels of one batch row (warp w
// takes channel d0 + w) and walks one chunk of the sequence in 32-step TMA tiles (the same maps
// and shared-memory layout as the serial kernel); lane t of a warp takes step t of the tile.
// Per tile and state n, each lane forms its step's pair e_t = (A_bar_t, B_bar_t x_t) and the warp
// runs an inclusive Kogge-Stone scan of the pairs over its 32 lanes with the operator
//   (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)      (the earlier element on the left),
// five rounds of two shuffles; lane t then holds the map h -> A_t h + B_t of steps 0..t of the
// tile and applies it to the state carried in from the previous tile (the last lane's state,
// broadcast by one more shuffle). Long sequences use the same chunk split and carry kernel as
// the serial path: the local pass runs this kernel without the readout.
//
// Cost: eleven shuffles per state and tile step against one update, and the shuffle unit of an
// SM issues one warp instruction per clock, so this path runs at about a tenth of the serial
// walk's speed on B300; it is kept for comparison and for callers that want the pages' form.
//
// Pages: "Mamba/SSM complete guide" section 5 `parallel_scan` (the combine of (A_bar, B_bar x)
// pairs; its printed combine order and omitted down-sweep are read as the operator above) and
// "論文解説: Mamba" "Hardware-Aware Parallel Scan" (the scan over the sequence kept on chip).
#include "scan_fast.cuh"

namespace ssm {
namespace fast {
namespace {

constexpr int kAssocThreads = kCh * 32;   // one warp per channel, one lane per tile step

// softplus(v) = max(v, 0) + log1p(e^-|v|) with the same log1p polynomial as softplus2.
__device__ __forceinline__ float softplus1(float v) {
    const float e = ex2_approx(-fabsf(v) * kLog2e);
    float q = kLog1pPoly[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) q = fmaf(e, q, kLog1pPoly[i]);
    return fmaf(e, q, fmaxf(v, 0.f));
}

template <int N, bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS, int MODE>
__global__ void __launch_bounds__(kAssocThreads, 1)
scan_assoc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap md,
                  const __grid_constant__ CUtensorMap mz, const __grid_constant__ CUtensorMap mB,
                  const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap my,
                  const FastParams p) {
    constexpr bool kReadout = MODE == kFull;
    constexpr bool kGate = GATE && kReadout;
    using Lay = Layout<N, BF16, kVarPlain, kGate, kReadout>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBars);

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int d0 = blockIdx.x * kCh, b = blockIdx.y, chunk = blockIdx.z;
    const int d = d0 + w;
    const bool dvalid = d < p.dim;
    const int64_t t_begin = (int64_t)chunk * p.chunk;
    const int64_t t_end = t_begin + p.chunk < p.seqlen ? t_begin + p.chunk : p.seqlen;
    const int64_t len = t_end - t_begin;
    const int ntiles = (int)((len + kT - 1) / kT);
    const int64_t state_elems = (int64_t)gridDim.y * p.dim * N;

    // initial state (the same in every lane): h0 or the carried state of this chunk; zero in
    // the local pass
    const float* hinit = nullptr;
    int64_t hinit_room = 0;
    if constexpr (kReadout) {
        if (p.carry) {
            hinit = p.carry + ((int64_t)chunk * gridDim.y + b) * p.dim * N;
            hinit_room = (int64_t)p.nchunks * state_elems - ((int64_t)chunk * gridDim.y + b) * p.dim * N;
        } else if (p.h0) {
            hinit = p.h0 + (int64_t)b * p.dim * N;
            hinit_room = state_elems - (int64_t)b * p.dim * N;
        }
    }
    float A2[N], hprev[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        A2[n] = 0.f;
        hprev[n] = 0.f;
        if (dvalid && idx_ok((int64_t)d * N + n, (int64_t)p.dim * N, p.status)) {
            A2[n] = p.A[(int64_t)d * N + n] * kLog2e;
            if (hinit && idx_ok((int64_t)d * N + n, hinit_room, p.status)) hprev[n] = hinit[(int64_t)d * N + n];
        }
    }
    const float bias = (dvalid && p.bias) ? p.bias[d] : 0.f;
    const float Dd = (DSKIP && dvalid) ? p.D[d] : 0.f;

    auto stage_ptr = [&](int buf) { return smem + Lay::kRing + buf * Lay::kStageStride; };
    auto issue = [&](int s) {
        const int buf = s % kStages;
        unsigned char* st = stage_ptr(buf);
        constexpr unsigned kBytes =
            Lay::kXBox + Lay::kTileX + (kGate ? Lay::kTileX : 0) + Lay::kTileB + (kReadout ? Lay::kTileB : 0);
        mbar_arrive_expect_tx(&bars[buf], kBytes);
        const int t0 = (int)(t_begin + (int64_t)s * kT);
        tma_load_3d(st, &mx, d0, t0, b, &bars[buf]);
        tma_load_3d(st + Lay::kOffD, &md, d0, t0, b, &bars[buf]);
        if constexpr (kGate) tma_load_3d(st + Lay::kOffZ, &mz, d0, t0, b, &bars[buf]);
        tma_load_3d(st + Lay::kOffB, &mB, 0, t0, b, &bars[buf]);
        if constexpr (kReadout) tma_load_3d(st + Lay::kOffC, &mC, 0, t0, b, &bars[buf]);
    };
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&mx);
        prefetch_tensormap(&mB);
        for (int s = p.skip_first_load ? 1 : 0; s < kStages && s < ntiles; ++s) issue(s);
    }
    __syncthreads();

    float dtsum = 0.f;   // local pass: this lane's share of the chunk's sum of dt
    bool failed = false;
    for (int s = 0; s < ntiles; ++s) {
        const int buf = s % kStages;
        const bool ok = mbar_wait_bounded(&bars[buf], (s / kStages) & 1, p.status);
        if (__syncthreads_or(!ok)) {
            // give up; first wait (bounded) for the later tiles already issued, so that no copy
            // still targets this CTA's shared memory
            if (tid == 0)
                for (int s2 = s + 1; s2 < s + kStages && s2 < ntiles; ++s2)
                    mbar_wait_bounded(&bars[s2 % kStages], (s2 / kStages) & 1, p.status);
            failed = true;
            break;
        }
        const unsigned char* st = stage_ptr(buf);
        const int rem = (int)(len - (int64_t)s * kT);
        const bool live = lane < (rem < kT ? rem : kT);   // rows past the chunk keep the state
        const float x = live ? ld_io(st, lane * kCh + w, BF16) : 0.f;
        float dt = 0.f;
        if (live) {
            const float v = ld_io(st + Lay::kOffD, lane * kCh + w, BF16) + bias;
            dt = SOFTPLUS ? softplus1(v) : v;
        }
        if constexpr (!kReadout) dtsum += dt;
        const float u = dt * x;
        float acc = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            float a = ex2_approx(dt * A2[n]);
            float bb = u * ld_io(st + Lay::kOffB, lane * N + n, BF16);
#pragma unroll
            for (int k = 1; k < 32; k <<= 1) {
                const float ap = __shfl_up_sync(0xffffffffu, a, k);
                const float bp = __shfl_up_sync(0xffffffffu, bb, k);
                if (lane >= k) {
                    bb = fmaf(a, bp, bb);   // later map after the earlier one: a b' + b
                    a *= ap;
                }
            }
            const float h = fmaf(a, hprev[n], bb);   // the state after this lane's step
            if constexpr (kReadout) acc = fmaf(ld_io(st + Lay::kOffC, lane * N + n, BF16), h, acc);
            hprev[n] = __shfl_sync(0xffffffffu, h, 31);
        }
        if constexpr (kReadout) {
            float y = acc;
            if constexpr (DSKIP) y = fmaf(Dd, x, y);
            if constexpr (kGate) y *= silu_fast(ld_io(st + Lay::kOffZ, lane * kCh + w, BF16));
            unsigned char* ys = smem + Lay::kY;
            if (s >= 1 && tid == 0) tma_store_wait_read<0>();   // the previous tile's store read ys
            __syncthreads();
            if constexpr (BF16)
                reinterpret_cast<__nv_bfloat16*>(ys)[lane * kCh + w] = __float2bfloat16_rn(y);
            else
                reinterpret_cast<float*>(ys)[lane * kCh + w] = y;
            fence_proxy_async_smem();
        }
        __syncthreads();   // every lane is done with this stage
        if (tid == 0) {
            if constexpr (kReadout) {
                tma_store_3d(&my, d0, (int)(t_begin + (int64_t)s * kT), b, smem + Lay::kY);
                tma_store_commit();
            }
            if (s + kStages < ntiles) issue(s + kStages);
        }
    }
    if (kReadout && tid == 0) tma_store_wait_all();
    if (failed || !dvalid) return;
    if constexpr (kReadout) {
        if (p.h_last && chunk == (int)gridDim.z - 1 && lane == 0) {
            const int64_t o = ((int64_t)b * p.dim + d) * N;
#pragma unroll
            for (int n = 0; n < N; ++n)
                if (idx_ok(o + n, state_elems, p.status)) p.h_last[o + n] = hprev[n];
        }
    } else {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dtsum += __shfl_xor_sync(0xffffffffu, dtsum, o);
        if (lane == 0) {
            const int64_t o = (((int64_t)(chunk + 1) * gridDim.y + b) * p.dim + d) * N;
#pragma unroll
            for (int n = 0; n < N; ++n)
                if (idx_ok(o + n, (int64_t)p.nchunks * state_elems, p.status)) p.carry[o + n] = hprev[n];
            const int64_t os = ((int64_t)chunk * gridDim.y + b) * p.dim + d;
            if (idx_ok(os, (int64_t)(p.nchunks - 1) * gridDim.y * p.dim, p.status)) p.sumdt[os] = dtsum;
        }
    }
}

template <int N, bool BF16, bool GATE, bool DSKIP, bool SOFTPLUS, int MODE>
cudaError_t launch_assoc_t(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                           cudaStream_t st) {
    using Lay = Layout<N, BF16, kVarPlain, GATE && MODE == kFull, MODE == kFull>;
    auto kern = scan_assoc_kernel<N, BF16, GATE, DSKIP, SOFTPLUS, MODE>;
    cudaError_t e = set_max_carveout_once<scan_assoc_kernel<N, BF16, GATE, DSKIP, SOFTPLUS, MODE>>(Lay::kTotal);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + kCh - 1) / kCh), (unsigned)a.batch, (unsigned)nz);
    kern<<<grid, kAssocThreads, Lay::kTotal, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], fp);
    note_launches(1);
    return cudaGetLastError();
}

template <int N, bool BF16, int MODE>
cudaError_t assoc_flags(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz, cudaStream_t st) {
    const bool gate = a.z != nullptr, dskip = a.D != nullptr, sp = a.softplus != 0;
    if constexpr (MODE == kPass1) {
        return sp ? launch_assoc_t<N, BF16, false, false, true, MODE>(maps, fp, a, nz, st)
                  : launch_assoc_t<N, BF16, false, false, false, MODE>(maps, fp, a, nz, st);
    } else {
#define SSM_ASSOC_CASE(G_, D_, S_) \
    if (gate == G_ && dskip == D_ && sp == S_) return launch_assoc_t<N, BF16, G_, D_, S_, MODE>(maps, fp, a, nz, st);
        SSM_ASSOC_CASE(true, true, true)
        SSM_ASSOC_CASE(true, true, false)
        SSM_ASSOC_CASE(true, false, true)
        SSM_ASSOC_CASE(true, false, false)
        SSM_ASSOC_CASE(false, true, true)
        SSM_ASSOC_CASE(false, true, false)
        SSM_ASSOC_CASE(false, false, true)
        SSM_ASSOC_CASE(false, false, false)
#undef SSM_ASSOC_CASE
    }
    return cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t assoc_dispatch(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz, cudaStream_t st) {
    const bool bf = a.io_bf16 != 0;
    switch (a.dstate) {
        case 16: return bf ? assoc_flags<16, true, MODE>(maps, fp, a, nz, st)
                           : assoc_flags<16, false, MODE>(maps, fp, a, nz, st);
        case 32: return bf ? assoc_flags<32, true, MODE>(maps, fp, a, nz, st)
                           : assoc_flags<32, false, MODE>(maps, fp, a, nz, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t dispatch_assoc_full(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                                cudaStream_t st) {
    return assoc_dispatch<kFull>(maps, fp, a, nz, st);
}

cudaError_t dispatch_assoc_pass1(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                                 cudaStream_t st) {
    return assoc_dispatch<kPass1>(maps, fp, a, nz, st);
}

}  // namespace fast
}  // namespace ssm
