// Causal depthwise conv1d along t with K <= 4 taps per channel, then optionally SiLU: the
// prologue of the Mamba block's x branch,
//   v[b,t,d] = bias[d] + sum_k weight[d,k] * xp[b, t+k, d]  (xp = x_prev then x along t),
//   y = silu(v) or v.
// Pages: "Mamba/SSM complete guide" section 5 `MambaBlock` (depthwise nn.Conv1d, kernel
// d_conv, padding d_conv - 1, output cut to the first L steps, then F.silu); "論文解説: Mamba"
// "Mambaブロックの全体構成" (a d_conv = 4 convolution followed by SiLU).
//
// The operation reads x once and writes y once, so it is bound by HBM bandwidth; the kernel
// streams tiles through shared memory with TMA so that many bytes are in flight without
// holding registers:
//  * a tile is kT = 32 steps x 256 bytes of channels (128 bf16 or 64 fp32) of one batch row;
//    its x box starts kHalo = 3 steps early (zero-filled before t = 0), so a tile carries the
//    window its first outputs need; y leaves through a TMA store of the 32 x 256-byte box;
//  * a CTA owns one channel slice (its taps stay in registers) and walks that slice's
//    (b, step-tile) tiles with a kStages-deep ring of x boxes; four CTAs per SM keep 16 boxes
//    (143 KB) in flight per SM;
//  * thread (word w, row group g) forms the outputs of the 4-byte column w (2 bf16 channels as
//    one packed fp32 pair, or 1 fp32 channel) for steps 8g .. 8g + 7 from 11 shared-memory
//    rows: consecutive threads read consecutive words (no bank conflicts).
// With x_prev, the first tile of a batch row takes its window from x_prev instead of the zero
// fill. Every mbarrier wait is bounded; a wait that runs out latches SSM_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 256;
constexpr int kT = 32;               // output steps per tile
constexpr int kHalo = 3;             // steps before the tile in its x box (the widest window)
constexpr int kRowBytes = 256;       // bytes of channels per tile row
constexpr int kWords = kRowBytes / 4;
constexpr int kRowsPerThread = kT / (kThreads / kWords);   // 8
constexpr int kStages = 4;
constexpr int kXBox = (kT + kHalo) * kRowBytes;            // 8960 bytes, a multiple of 128
constexpr int kYBox = kT * kRowBytes;
constexpr int kSmem = kStages * kXBox + 2 * kYBox + 64;
constexpr int kCtasPerSm = 4;

struct ConvParams {
    int64_t batch, L, dim;
    int K;
    int rowtiles;           // ceil(L / kT)
    const float* w;         // (D, K)
    const float* bias;      // (D) or nullptr
    const void* x_prev;     // (b, K-1, D) or nullptr
    unsigned* status;
};

template <bool BF16>
__device__ __forceinline__ void widen_word(uint32_t v, float (&f)[BF16 ? 2 : 1]) {
    if constexpr (BF16) {
        f[0] = __uint_as_float(v << 16);
        f[1] = __uint_as_float(v & 0xffff0000u);
    } else {
        f[0] = __uint_as_float(v);
    }
}

template <bool BF16, bool SILU>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
conv1d_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap my, const ConvParams p) {
    constexpr int E = BF16 ? 2 : 1;            // channels per 4-byte word
    constexpr int kEsz = BF16 ? 2 : 4;
    constexpr int kChan = kRowBytes / kEsz;    // channels per slice
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    unsigned char* ybuf = smem + kStages * kXBox;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kXBox + 2 * kYBox);

    const int tid = threadIdx.x;
    const int word = tid % kWords, grp = tid / kWords;
    const int slice = blockIdx.x;
    const int64_t ntiles = p.batch * p.rowtiles;
    // this CTA's tiles: blockIdx.y, blockIdx.y + gridDim.y, ...
    const int64_t mine = ntiles > blockIdx.y ? (ntiles - blockIdx.y + gridDim.y - 1) / gridDim.y : 0;

    // taps of this thread's channels, right-aligned: w4[e][3] multiplies x_t
    const int64_t c0 = (int64_t)slice * kChan + word * E;
    float w4[E][4], bv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int64_t c = c0 + e;
        bv[e] = (c < p.dim && p.bias && idx_ok(c, p.dim, p.status)) ? p.bias[c] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = j - (4 - p.K);
            w4[e][j] = (c < p.dim && k >= 0 && idx_ok(c * p.K + k, p.dim * p.K, p.status)) ? p.w[c * p.K + k] : 0.f;
        }
    }

    auto tile_coords = [&](int64_t i, int& b, int& t0) {
        const int64_t j = blockIdx.y + i * gridDim.y;
        b = (int)(j / p.rowtiles);
        t0 = (int)(j % p.rowtiles) * kT;
    };
    auto issue = [&](int64_t i) {
        int b, t0;
        tile_coords(i, b, t0);
        uint64_t* bar = &bars[i % kStages];
        mbar_arrive_expect_tx(bar, kXBox);
        tma_load_3d(ring + (i % kStages) * kXBox, &mx, slice * kChan, t0 - kHalo, b, bar);
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        prefetch_tensormap(&mx);
        prefetch_tensormap(&my);
        for (int64_t i = 0; i < kStages && i < mine; ++i) issue(i);
    }
    __syncthreads();

    for (int64_t i = 0; i < mine; ++i) {
        const int s = (int)(i % kStages);
        const bool ok = mbar_wait_bounded(&bars[s], (unsigned)((i / kStages) & 1), p.status);
        if (tid == 0 && i >= 2) tma_store_wait_read<1>();   // the store of tile i-2 has left its buffer
        if (__syncthreads_or(!ok)) {
            // give up; wait (bounded) for the loads still in flight into this CTA's memory
            if (tid == 0)
                for (int64_t i2 = i + 1; i2 < i + kStages && i2 < mine; ++i2)
                    mbar_wait_bounded(&bars[i2 % kStages], (unsigned)((i2 / kStages) & 1), p.status);
            break;
        }
        int b, t0;
        tile_coords(i, b, t0);
        const uint32_t* xs = reinterpret_cast<const uint32_t*>(ring + s * kXBox);
        uint32_t* ys = reinterpret_cast<uint32_t*>(ybuf + (i & 1) * kYBox);
        // box row r holds step t0 - kHalo + r; this thread's outputs are rows kHalo + r0 + q
        const int r0 = kRowsPerThread * grp;
        float win[3][E];
        if (grp == 0 && t0 == 0 && p.x_prev) {
#pragma unroll
            for (int m = 3; m >= 1; --m)   // x_{-m}
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int64_t c = c0 + e;
                    float v = 0.f;
                    if (m <= p.K - 1 && c < p.dim) {
                        const int64_t ip = ((int64_t)b * (p.K - 1) + (p.K - 1 - m)) * p.dim + c;
                        if (idx_ok(ip, p.batch * (p.K - 1) * p.dim, p.status)) v = load_f32(p.x_prev, ip, BF16);
                    }
                    win[3 - m][e] = v;
                }
        } else {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                float f[E];
                widen_word<BF16>(xs[(r0 + j) * kWords + word], f);
#pragma unroll
                for (int e = 0; e < E; ++e) win[j][e] = f[e];
            }
        }
        if constexpr (BF16) {
            // the word's two channels as one packed pair through the taps and SiLU
            f2 W[4], Bv = pk(bv[0], bv[1]), X[3];
#pragma unroll
            for (int j = 0; j < 4; ++j) W[j] = pk(w4[0][j], w4[1][j]);
#pragma unroll
            for (int j = 0; j < 3; ++j) X[j] = pk(win[j][0], win[j][1]);
            const f2 kNegLog2e = pk(-kLog2e, -kLog2e), kOne = pk(1.f, 1.f);
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q) {
                const uint32_t raw = xs[(r0 + kHalo + q) * kWords + word];
                const f2 xv = pk(__uint_as_float(raw << 16), __uint_as_float(raw & 0xffff0000u));
                f2 v = fma2(W[3], xv, Bv);
                v = fma2(W[2], X[2], v);
                v = fma2(W[1], X[1], v);
                v = fma2(W[0], X[0], v);
                X[0] = X[1];
                X[1] = X[2];
                X[2] = xv;
                float lo, hi;
                if constexpr (SILU) {
                    // silu(v) = v / (1 + 2^(-v log2 e)) from the SFU's ex2 and rcp (a few ulp)
                    float e0, e1;
                    upk(mul2(v, kNegLog2e), e0, e1);
                    const f2 den = fma2(kOne, pk(ex2_approx(e0), ex2_approx(e1)), kOne);
                    float d0, d1;
                    upk(den, d0, d1);
                    upk(mul2(v, pk(rcp_approx(d0), rcp_approx(d1))), lo, hi);
                } else {
                    upk(v, lo, hi);
                }
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
                ys[(r0 + q) * kWords + word] = *reinterpret_cast<const uint32_t*>(&h2);
            }
        } else {
#pragma unroll
            for (int q = 0; q < kRowsPerThread; ++q) {
                float xv[E];
                widen_word<BF16>(xs[(r0 + kHalo + q) * kWords + word], xv);
                float v = fmaf(w4[0][3], xv[0], bv[0]);
                v = fmaf(w4[0][2], win[2][0], v);
                v = fmaf(w4[0][1], win[1][0], v);
                v = fmaf(w4[0][0], win[0][0], v);
                win[0][0] = win[1][0];
                win[1][0] = win[2][0];
                win[2][0] = xv[0];
                // silu from the SFU's ex2 and rcp (a few ulp)
                ys[(r0 + q) * kWords + word] = __float_as_uint(SILU ? silu_fast(v) : v);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();   // ring slot s read, the y buffer written
        if (tid == 0) {
            tma_store_3d(&my, slice * kChan, t0, b, ys);
            tma_store_commit();
            if (i + kStages < mine) issue(i + kStages);
        }
    }
    if (tid == 0) tma_store_wait_all();
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// 3-D map over a contiguous (b, L, D) tensor: dims (D, L, b), box (256 bytes of channels, rows, 1).
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t D, int64_t L, int64_t b, int rows) {
    auto fn = encoder();
    if (!fn) return false;
    const int64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)b};
    cuuint64_t strides[2] = {(cuuint64_t)(D * esz), (cuuint64_t)(L * D * esz)};
    cuuint32_t box[3] = {(cuuint32_t)(kRowBytes / esz), (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BF16, bool SILU>
cudaError_t launch_t(const CUtensorMap& mx, const CUtensorMap& my, const ConvParams& p, int nslices, int per_slice,
                     cudaStream_t st) {
    auto kern = conv1d_kernel<BF16, SILU>;
    cudaError_t e = set_smem_once<conv1d_kernel<BF16, SILU>>(kSmem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)nslices, (unsigned)per_slice), kThreads, kSmem, st>>>(mx, my, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv1d(const Conv1dArgs& a, cudaStream_t st) {
    const bool bf = a.io_bf16 != 0;
    const int64_t esz = bf ? 2 : 4;
    const int64_t chan = kRowBytes / esz;
    if (a.batch > INT32_MAX || a.seqlen > INT32_MAX - 2 * kT || a.dim > INT32_MAX) return cudaErrorInvalidValue;
    CUtensorMap mx, my;
    if (!make_map(&mx, a.x, bf, a.dim, a.seqlen, a.batch, kT + kHalo) ||
        !make_map(&my, a.y, bf, a.dim, a.seqlen, a.batch, kT))
        return cudaErrorInvalidValue;
    ConvParams p;
    p.batch = a.batch;
    p.L = a.seqlen;
    p.dim = a.dim;
    p.K = a.k;
    p.rowtiles = (int)((a.seqlen + kT - 1) / kT);
    p.w = a.w;
    p.bias = a.bias;
    p.x_prev = a.x_prev;
    p.status = a.status;
    if (!p.status) return cudaErrorInvalidValue;
    const int64_t nslices = (a.dim + chan - 1) / chan;
    if (nslices > INT32_MAX) return cudaErrorInvalidValue;
    const int64_t ntiles = a.batch * p.rowtiles;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // one wave of CTAs: the slices share the SMs' kCtasPerSm slots
    int64_t per_slice = (int64_t)sms * kCtasPerSm / nslices;
    if (per_slice < 1) per_slice = 1;
    if (per_slice > ntiles) per_slice = ntiles;
    if (per_slice > 65535) per_slice = 65535;
    if (a.silu)
        return bf ? launch_t<true, true>(mx, my, p, (int)nslices, (int)per_slice, st)
                  : launch_t<false, true>(mx, my, p, (int)nslices, (int)per_slice, st);
    return bf ? launch_t<true, false>(mx, my, p, (int)nslices, (int)per_slice, st)
              : launch_t<false, false>(mx, my, p, (int)nslices, (int)per_slice, st);
}

}  // namespace ssm
