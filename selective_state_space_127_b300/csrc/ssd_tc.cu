// Mamba-2 SSD chunked scan on the fifth-generation tensor cores (tcgen05), for bf16 I/O with
// head dimension P = 64 and state size N = 128.
//
// One CTA (256 threads) per (batch, head) walks the sequence in blocks of Q = 128 steps;
// the N x P state S stays on chip (fp32 registers, two threads per row n, plus a bf16 copy
// in shared memory as an MMA operand). Per block, with cum_t the inclusive cumulative sum of
// dt A_h inside the block (the decay from the block start to step t):
//
//   G      = C B^T                                  (Q x Q, K = N)      tcgen05, TMEM
//   M[t,s] = G[t,s] exp(cum_t - cum_s) dt_s, s <= t; 0 above the diagonal
//   Y      = M X + (exp(cum) o C) S_prev           (Q x P, K = Q + N)  tcgen05, M from TMEM
//   y_t    = Y_t (+ D x_t) (* silu z_t)
//   S      = exp(cum_last) S_prev + (w o B)^T X,    w_s = exp(cum_last - cum_s) dt_s
//                                                   (N x P, K = Q)      tcgen05
//
// which is the block decomposition of the semiseparable matrix of the recurrence
// S_t = exp(dt_t A_h) S_{t-1} + dt_t B_t x_t^T, y_t = S_t^T C_t: diagonal blocks as masked
// matrix products, the hand-off between blocks through the state (a rank-N product).
// A chunk of Q' = 128 k steps (the chunk length the caller asks for) is computed as k such
// blocks; the result does not depend on the chunk length beyond rounding.
//
// Data movement: TMA (4-D maps, 128-byte swizzle) brings the C and B blocks (128 x 128) and
// the x block (128 x 64) into shared memory in the layouts the MMAs read directly (C and B
// K-major for G; C, rescaled in place by exp(cum_t), K-major for the hand-off; B, rescaled
// in place by w_s, as the MN-major A operand of the state product; x MN-major as the B
// operand); the y block leaves by TMA store from the x buffer. The next block's C and B are
// requested as soon as this block's products are done with them, its x once y has left.
// Tensor memory: G (128 columns, then the state product), M in bf16 (64) and Y (64): 256
// columns, so two CTAs share an SM. Eight warps: two per TMEM lane quarter (the rows a warp
// may access), splitting the columns of the mask, scaling and epilogue work between them.
// One thread issues the MMAs and waits for them; the others wait at the CTA barrier.
//
// Pages: "Mamba-2 / Structured State Space Duality" (abeam) "基本アイデア" (SSM as a
// semiseparable matrix; diagonal blocks by ordinary matrix products, off-diagonal blocks by a
// low-rank hand-off of the state) and "線形形式と二次形式を使い分ける"; "Mamba/SSM complete
// guide" section 6 "SSD演算の概念" (intra-chunk matrix products on tensor cores, inter-chunk
// state recurrence) and `Mamba2Block` (one A per head, B and C shared by the heads of a group).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kQ = 128;          // steps per block
constexpr int kP = 64;           // head dimension
constexpr int kN = 128;          // state size
constexpr int kThreads = 256;    // 8 warps: two per TMEM lane quarter, splitting the columns
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColG = 0;    // G (128 columns); after the mask pass the state product (0..63)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColM = 128;  // M in bf16 pairs (64 columns)
constexpr uint32_t kColY = 192;  // Y = M X + (exp(cum) o C) S_prev (64 columns)

constexpr int kAtom = 16384;     // 128 rows x 128 bytes
constexpr int kSmC = 0;
constexpr int kSmB = 2 * kAtom;
constexpr int kSmX = 4 * kAtom;
constexpr int kSmS = 5 * kAtom;
constexpr int kSmCs = 6 * kAtom;             // float [kQ]: cum_t log2(e)
constexpr int kSmLw = kSmCs + kQ * 4;        // float [kQ]: dt_s
constexpr int kSmEv = kSmLw + kQ * 4;        // float [kQ]: exp(cum_t)
constexpr int kSmWv = kSmEv + kQ * 4;        // float [kQ]: exp(cum_last - cum_s) dt_s
constexpr int kSmRed = kSmWv + kQ * 4;       // float [8]: warp totals of the scan, exp(cum_last)
constexpr int kSmBar = kSmRed + 64;          // 4 mbarriers: C, B and x loads, MMA completion
constexpr int kSmTmem = kSmBar + 32;         // tensor-memory base address
constexpr int kSmemUsed = kSmTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024; // room to align the base to 1024 bytes

constexpr uint32_t kIdescG = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescY = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdescS = tc::idesc_bf16(128, 64, true, true);

struct TcParams {
    int64_t seqlen;
    int nheads;
    int heads_per_group;
    int nblocks;
    int softplus;
    const void* x;         // (b, L, H, P) bf16, for the D skip
    const void* delta;     // (b, L, H) bf16
    const float* A;
    const float* D;
    const void* z;         // (b, L, H, P) bf16 or NULL
    const float* bias;
    const float* h0;       // (b, H, N, P) fp32 or NULL
    float* h_last;         // (b, H, N, P) fp32 or NULL
    unsigned* status;
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                             const void* src) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Eight bf16 values (16 bytes) times a scalar held as a packed pair, rounded back to bf16.
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, f2 s2) {
    float a, c;
    uint4 r;
    upk(mul2(pk(bf_lo(v.x), bf_hi(v.x)), s2), a, c);
    r.x = tc::pack_bf16(a, c);
    upk(mul2(pk(bf_lo(v.y), bf_hi(v.y)), s2), a, c);
    r.y = tc::pack_bf16(a, c);
    upk(mul2(pk(bf_lo(v.z), bf_hi(v.z)), s2), a, c);
    r.z = tc::pack_bf16(a, c);
    upk(mul2(pk(bf_lo(v.w), bf_hi(v.w)), s2), a, c);
    r.w = tc::pack_bf16(a, c);
    return r;
}

__global__ void __launch_bounds__(kThreads, 2)
ssd_tc_kernel(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mB,
              const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap mY, const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
    unsigned char* sC = sm + kSmC;
    unsigned char* sB = sm + kSmB;
    unsigned char* sX = sm + kSmX;
    unsigned char* sS = sm + kSmS;
    float* cs = reinterpret_cast<float*>(sm + kSmCs);    // cum_t log2 e
    float* lw = reinterpret_cast<float*>(sm + kSmLw);    // dt_s
    float* ev = reinterpret_cast<float*>(sm + kSmEv);    // exp(cum_t)
    float* wv = reinterpret_cast<float*>(sm + kSmWv);    // exp(cum_last - cum_s) dt_s
    float* red = reinterpret_cast<float*>(sm + kSmRed);
    uint64_t* bar_c = reinterpret_cast<uint64_t*>(sm + kSmBar);
    uint64_t* bar_b = bar_c + 1;
    uint64_t* bar_x = bar_c + 2;
    uint64_t* bar_mma = bar_c + 3;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kSmTmem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;        // the TMEM lanes (rows) this warp can access
    const int half = warp >> 2;          // which half of the columns (or atom) it takes
    const int row = tid & 127;           // = 32 quarter + lane
    const int h = blockIdx.x, b = blockIdx.y;
    const int grp = h / p.heads_per_group;
    const int64_t L = p.seqlen;
    const int H = p.nheads;

    if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (tid == 0) {
        mbar_init(bar_c, 1);
        mbar_init(bar_b, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tensormap(&mX);
        prefetch_tensormap(&mB);
        prefetch_tensormap(&mC);
        prefetch_tensormap(&mY);
    }

    // the state: row `row`, columns [32 half, 32 half + 32) in fp32 registers; its bf16 copy
    // (the B operand of the hand-off product) in sS
    float S[kP / 2];
    {
        const float* src = p.h0 ? p.h0 + (((int64_t)b * H + h) * kN + row) * kP + 32 * half : nullptr;
#pragma unroll
        for (int i = 0; i < kP / 2; i += 4) {
            const float4 v = src ? *reinterpret_cast<const float4*>(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            S[i] = v.x;
            S[i + 1] = v.y;
            S[i + 2] = v.z;
            S[i + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 v;
            v.x = tc::pack_bf16(S[8 * j], S[8 * j + 1]);
            v.y = tc::pack_bf16(S[8 * j + 2], S[8 * j + 3]);
            v.z = tc::pack_bf16(S[8 * j + 4], S[8 * j + 5]);
            v.w = tc::pack_bf16(S[8 * j + 6], S[8 * j + 7]);
            *reinterpret_cast<uint4*>(sS + sw128(row, 4 * half + j)) = v;
        }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);

    const float Ah = p.A[h];
    const float bias = p.bias ? p.bias[h] : 0.f;
    const float Dh = p.D ? p.D[h] : 0.f;
    const uint32_t aC = smem_u32(sC), aB = smem_u32(sB), aX = smem_u32(sX), aS = smem_u32(sS);
    const __nv_bfloat16* delta = static_cast<const __nv_bfloat16*>(p.delta);

    // Load schedule: C and B of block j+1 once the products of block j are done with them,
    // x of block j+1 once the y of block j (staged in the x buffer) has been read out by its
    // TMA store.
    auto load_c = [&](int j) {
        mbar_arrive_expect_tx(bar_c, 2 * kAtom);
        tma_load_4d(sC, &mC, 0, grp, j * kQ, b, bar_c);
        tma_load_4d(sC + kAtom, &mC, 64, grp, j * kQ, b, bar_c);
    };
    auto load_b = [&](int j) {
        mbar_arrive_expect_tx(bar_b, 2 * kAtom);
        tma_load_4d(sB, &mB, 0, grp, j * kQ, b, bar_b);
        tma_load_4d(sB + kAtom, &mB, 64, grp, j * kQ, b, bar_b);
    };
    auto load_x = [&](int j) {
        mbar_arrive_expect_tx(bar_x, kAtom);
        tma_load_4d(sX, &mX, 0, h, j * kQ, b, bar_x);
    };
    if (tid == 0 && p.nblocks > 0) {
        load_c(0);
        load_b(0);
        load_x(0);
    }
    // delta of row t (threads of the first warpgroup), one block ahead
    auto load_delta = [&](int j) -> float {
        const int64_t tt = (int64_t)j * kQ + row;
        return (half == 0 && j < p.nblocks && tt < L) ? __bfloat162float(delta[((int64_t)b * L + tt) * H + h]) : 0.f;
    };
    float draw_next = load_delta(0);

    unsigned ph_mma = 0;
    bool failed = false;
    for (int j = 0; j < p.nblocks; ++j) {
        const int t0 = j * kQ;
        const unsigned ph_ld = j & 1;
        const int64_t t = t0 + row;
        // dt_t and the inclusive cumulative sum of dt A_h over the block (first warpgroup, row t)
        if (half == 0) {
            float dt = 0.f;
            if (t < L) {
                const float v = draw_next + bias;
                dt = p.softplus ? softplus_accurate(v) : v;
            }
            float cum = dt * Ah;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, cum, o);
                if (lane >= o) cum += n;
            }
            if (lane == 31) red[warp] = cum;
            cs[row] = cum;   // provisional: the warp-local prefix, completed below
            lw[row] = dt;
        }
        draw_next = load_delta(j + 1);
        __syncthreads();
        if (half == 0) {
            float before = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (w < warp) before += red[w];
            const float cum = cs[row] + before;
            const float dt = lw[row];
            const float cum_last = red[0] + red[1] + red[2] + red[3];
            const float cs_t = cum * kLog2e;
            cs[row] = cs_t;
            lw[row] = dt;
            ev[row] = ex2_approx(cs_t);
            wv[row] = ex2_approx((cum_last - cum) * kLog2e) * dt;
            if (row == 0) red[4] = ex2_approx(cum_last * kLog2e);
        }

        // G = C B^T (one thread issues and waits; the others wait at the barrier)
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait_bounded(bar_c, ph_ld, p.status) && mbar_wait_bounded(bar_b, ph_ld, p.status);
            if (ok) {
                tc::fence_after_sync();
#pragma unroll
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t off = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_ss(tmem + kColG, tc::sdesc_sw128(aC + off, 16, 1024),
                               tc::sdesc_sw128(aB + off, 16, 1024), kIdescG, k > 0);
                }
                tc::commit(bar_mma);
                ok = mbar_wait_bounded(bar_mma, ph_mma, p.status);
            }
        }
        ph_mma ^= 1;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc::fence_after_sync();
        const float cs_t = cs[row];
        const float e_last = red[4];

        // G has read C and B: scale them in place, row t of C by exp(cum_t) (the decay from the
        // block start, so that (exp(cum) o C) S_prev is the state hand-off) and row s of B by
        // w_s = exp(cum_last - cum_s) dt_s (the weights of the state product (w o B)^T X).
        // Thread (row, half) takes atom `half` of the row; the chunks are walked in swizzled
        // order so that eight consecutive rows hit eight different bank groups.
        {
            const f2 e2 = pk(ev[row], ev[row]);
            const f2 w2 = pk(wv[row], wv[row]);
            uint4* rowc = reinterpret_cast<uint4*>(sC + half * kAtom + row * 128);
            uint4* rowb = reinterpret_cast<uint4*>(sB + half * kAtom + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = i ^ (row & 7);
                rowc[c] = scale_bf16x8(rowc[c], e2);
                rowb[c] = scale_bf16x8(rowb[c], w2);
            }
        }
        // M[t, s] = G[t, s] exp(cum_t - cum_s) dt_s for s <= t (bf16 pairs in columns kColM..):
        // warp (quarter, half) takes the 32-column chunks kc = half and half + 2 of its rows
#pragma unroll
        for (int ic = 0; ic < 2; ++ic) {
            const int kc = half + 2 * ic;
            uint32_t packed[16];
            if (kc < quarter) {          // below the diagonal: every s < t
                uint32_t r[32];
                tc::ld32(lane_base + kColG + 32 * kc, r);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(cs + 32 * kc + i);
                    const float4 d4 = *reinterpret_cast<const float4*>(lw + 32 * kc + i);
                    packed[i / 2] = tc::pack_bf16(__uint_as_float(r[i]) * d4.x * ex2_approx(cs_t - c4.x),
                                                  __uint_as_float(r[i + 1]) * d4.y * ex2_approx(cs_t - c4.y));
                    packed[i / 2 + 1] = tc::pack_bf16(__uint_as_float(r[i + 2]) * d4.z * ex2_approx(cs_t - c4.z),
                                                      __uint_as_float(r[i + 3]) * d4.w * ex2_approx(cs_t - c4.w));
                }
            } else if (kc == quarter) {  // the diagonal chunk: s <= t
                uint32_t r[32];
                tc::ld32(lane_base + kColG + 32 * kc, r);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(cs + 32 * kc + i);
                    const float4 d4 = *reinterpret_cast<const float4*>(lw + 32 * kc + i);
                    const float m0 = i <= lane ? __uint_as_float(r[i]) * d4.x * ex2_approx(cs_t - c4.x) : 0.f;
                    const float m1 = i + 1 <= lane ? __uint_as_float(r[i + 1]) * d4.y * ex2_approx(cs_t - c4.y) : 0.f;
                    const float m2 = i + 2 <= lane ? __uint_as_float(r[i + 2]) * d4.z * ex2_approx(cs_t - c4.z) : 0.f;
                    const float m3 = i + 3 <= lane ? __uint_as_float(r[i + 3]) * d4.w * ex2_approx(cs_t - c4.w) : 0.f;
                    packed[i / 2] = tc::pack_bf16(m0, m1);
                    packed[i / 2 + 1] = tc::pack_bf16(m2, m3);
                }
            } else {                     // above the diagonal
#pragma unroll
                for (int i = 0; i < 16; ++i) packed[i] = 0u;
            }
            tc::st16(lane_base + kColM + 16 * kc, packed);
        }
        tc::wait_st();
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // Y = M X + (exp(cum) o C) S_prev and S_acc = (w o B)^T X (S_acc over G's columns)
        if (tid == 0) {
            ok = mbar_wait_bounded(bar_x, ph_ld, p.status);
            if (ok) {
                tc::fence_after_sync();
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    tc::mma_ts(tmem + kColY, tmem + kColM + 8 * k, tc::sdesc_sw128(aX + k * 2048, kAtom, 1024),
                               kIdescY, k > 0);
#pragma unroll
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t off = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_ss(tmem + kColY, tc::sdesc_sw128(aC + off, 16, 1024),
                               tc::sdesc_sw128(aS + k * 2048, kAtom, 1024), kIdescY, 1);
                }
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    tc::mma_ss(tmem + kColS, tc::sdesc_sw128(aB + k * 2048, kAtom, 1024),
                               tc::sdesc_sw128(aX + k * 2048, kAtom, 1024), kIdescS, k > 0);
                tc::commit(bar_mma);
                ok = mbar_wait_bounded(bar_mma, ph_mma, p.status);
            }
            // C and B of this block are no longer read
            if (ok && j + 1 < p.nblocks) {
                load_c(j + 1);
                load_b(j + 1);
            }
        }
        ph_mma ^= 1;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc::fence_after_sync();

        // epilogue: y row t, columns [32 half, +32) into sX (free now); the state row, same
        // columns; 16 columns at a time
        const __nv_bfloat16* xrow = p.D && t < L ? static_cast<const __nv_bfloat16*>(p.x) +
                                                       (((int64_t)b * L + t) * H + h) * kP + 32 * half
                                                 : nullptr;
        const __nv_bfloat16* zrow = p.z && t < L ? static_cast<const __nv_bfloat16*>(p.z) +
                                                       (((int64_t)b * L + t) * H + h) * kP + 32 * half
                                                 : nullptr;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t ry[16];
            tc::ld16(lane_base + kColY + 32 * half + 16 * q, ry);
            tc::wait_ld();
            float yv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) yv[i] = __uint_as_float(ry[i]);
            if (xrow) {
#pragma unroll
                for (int i = 0; i < 16; i += 8) {
                    const uint4 v = *reinterpret_cast<const uint4*>(xrow + 16 * q + i);
                    yv[i] = fmaf(Dh, bf_lo(v.x), yv[i]);
                    yv[i + 1] = fmaf(Dh, bf_hi(v.x), yv[i + 1]);
                    yv[i + 2] = fmaf(Dh, bf_lo(v.y), yv[i + 2]);
                    yv[i + 3] = fmaf(Dh, bf_hi(v.y), yv[i + 3]);
                    yv[i + 4] = fmaf(Dh, bf_lo(v.z), yv[i + 4]);
                    yv[i + 5] = fmaf(Dh, bf_hi(v.z), yv[i + 5]);
                    yv[i + 6] = fmaf(Dh, bf_lo(v.w), yv[i + 6]);
                    yv[i + 7] = fmaf(Dh, bf_hi(v.w), yv[i + 7]);
                }
            }
            if (zrow) {
#pragma unroll
                for (int i = 0; i < 16; i += 8) {
                    const uint4 v = *reinterpret_cast<const uint4*>(zrow + 16 * q + i);
                    yv[i] *= silu_accurate(bf_lo(v.x));
                    yv[i + 1] *= silu_accurate(bf_hi(v.x));
                    yv[i + 2] *= silu_accurate(bf_lo(v.y));
                    yv[i + 3] *= silu_accurate(bf_hi(v.y));
                    yv[i + 4] *= silu_accurate(bf_lo(v.z));
                    yv[i + 5] *= silu_accurate(bf_hi(v.z));
                    yv[i + 6] *= silu_accurate(bf_lo(v.w));
                    yv[i + 7] *= silu_accurate(bf_hi(v.w));
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint4 v;
                v.x = tc::pack_bf16(yv[8 * c], yv[8 * c + 1]);
                v.y = tc::pack_bf16(yv[8 * c + 2], yv[8 * c + 3]);
                v.z = tc::pack_bf16(yv[8 * c + 4], yv[8 * c + 5]);
                v.w = tc::pack_bf16(yv[8 * c + 6], yv[8 * c + 7]);
                *reinterpret_cast<uint4*>(sX + sw128(row, 4 * half + 2 * q + c)) = v;
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t rs[16];
            tc::ld16(lane_base + kColS + 32 * half + 16 * q, rs);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) S[16 * q + i] = fmaf(e_last, S[16 * q + i], __uint_as_float(rs[i]));
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint4 v;
                v.x = tc::pack_bf16(S[16 * q + 8 * c], S[16 * q + 8 * c + 1]);
                v.y = tc::pack_bf16(S[16 * q + 8 * c + 2], S[16 * q + 8 * c + 3]);
                v.z = tc::pack_bf16(S[16 * q + 8 * c + 4], S[16 * q + 8 * c + 5]);
                v.w = tc::pack_bf16(S[16 * q + 8 * c + 6], S[16 * q + 8 * c + 7]);
                *reinterpret_cast<uint4*>(sS + sw128(row, 4 * half + 2 * q + c)) = v;
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tma_store_4d(&mY, 0, h, t0, b, sX);
            tma_store_commit();
            if (j + 1 < p.nblocks) {
                tma_store_wait_read<0>();   // y has left the x buffer
                load_x(j + 1);
            }
        }
    }
    if (tid == 0) tma_store_wait_all();
    if (!failed && p.h_last) {
        float* dst = p.h_last + (((int64_t)b * H + h) * kN + row) * kP + 32 * half;
#pragma unroll
        for (int i = 0; i < kP / 2; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn4() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// 4-D bf16 map over a contiguous (d3, d2, d1, d0) tensor, box {64, 1, 128, 1}, 128-byte swizzle.
bool make_map4(CUtensorMap* m, const void* base, int64_t d0, int64_t d1, int64_t d2, int64_t d3) {
    auto fn = encode_fn4();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2, (cuuint64_t)d3};
    cuuint64_t strides[3] = {(cuuint64_t)(d0 * 2), (cuuint64_t)(d0 * d1 * 2), (cuuint64_t)(d0 * d1 * d2 * 2)};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

}  // namespace

bool ssd_tc_supported(const SSDArgs& a) {
    if (!a.io_bf16 || a.headdim != kP || a.dstate != kN) return false;
    if (a.chunk % kQ != 0) return false;
    if (a.nheads > 65535 || a.batch > 65535 || a.seqlen > ((int64_t)1 << 30)) return false;
    if (!al16(a.x) || !al16(a.B) || !al16(a.C) || !al16(a.y)) return false;
    if (a.z && !al16(a.z)) return false;
    if (a.h0 && !al16(a.h0)) return false;
    if (a.h_last && !al16(a.h_last)) return false;
    return encode_fn4() != nullptr;
}

cudaError_t launch_ssd_tc(const SSDArgs& a, cudaStream_t st) {
    CUtensorMap mX, mB, mC, mY;
    if (!make_map4(&mX, a.x, kP, a.nheads, a.seqlen, a.batch) ||
        !make_map4(&mB, a.B, kN, a.ngroups, a.seqlen, a.batch) ||
        !make_map4(&mC, a.C, kN, a.ngroups, a.seqlen, a.batch) ||
        !make_map4(&mY, a.y, kP, a.nheads, a.seqlen, a.batch))
        return cudaErrorInvalidValue;
    TcParams p;
    p.seqlen = a.seqlen;
    p.nheads = (int)a.nheads;
    p.heads_per_group = (int)(a.nheads / a.ngroups);
    p.nblocks = (int)((a.seqlen + kQ - 1) / kQ);
    p.softplus = a.softplus;
    p.x = a.x;
    p.delta = a.delta;
    p.A = a.A;
    p.D = a.D;
    p.z = a.z;
    p.bias = a.bias;
    p.h0 = a.h0;
    p.h_last = a.h_last;
    p.status = device_status_ptr();
    if (!p.status) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(ssd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.nheads, (unsigned)a.batch);
    ssd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mX, mB, mC, mY, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
