// Mamba-2 SSD chunked scan on the fifth-generation tensor cores (tcgen05), for bf16 I/O with
// head dimension P = 64 and state size N = 128.
//
// One CTA per (batch, head) walks the sequence in blocks of Q = 128 steps; the N x P state S
// stays on chip (fp32 registers, two threads per row n, plus a bf16 copy in shared memory as
// an MMA operand). Per block, with cum_t the inclusive cumulative sum of dt A_h inside the
// block (the decay from the block start to step t):
//
//   G      = C B^T                                  (Q x Q, K = N)      tcgen05, TMEM
//   M[t,s] = G[t,s] exp(cum_t - cum_s) dt_s, s <= t; 0 above the diagonal
//   Y      = M X                                    (Q x P, K = Q)      tcgen05, M from TMEM
//   Yoff   = C S_prev                               (Q x P, K = N)      tcgen05
//   y_t    = Y_t + exp(cum_t) Yoff_t  (+ D x_t) (* silu z_t)
//   S      = exp(cum_last) S_prev + B^T (w o X),    w_s = exp(cum_last - cum_s) dt_s
//                                                   (N x P, K = Q)      tcgen05
//
// which is the block decomposition of the semiseparable matrix of the recurrence
// S_t = exp(dt_t A_h) S_{t-1} + dt_t B_t x_t^T, y_t = S_t^T C_t: diagonal blocks as masked
// matrix products, the hand-off between blocks through the state (a rank-N product).
// A chunk of Q' = 128 k steps (the chunk length the caller asks for) is computed as k such
// blocks; the result does not depend on the chunk length beyond rounding.
//
// Pipeline. A control warp issues the TMA loads, the MMAs and the y stores; eight math warps
// (two per TMEM lane quarter, each taking the same half of every 32-column chunk of the mask,
// so both carry the same mix of factored, diagonal and zero columns) run the block scan of dt A,
// the mask,
// the scaled copy w o X and the epilogue. Below the diagonal the mask's decay is factored per
// 32-step chunk, exp(cum_t - cum_s) = exp(cum_t - cum_ref) exp(cum_ref - cum_s) with cum_ref
// the chunk's last step (both factors <= 1), so those elements need no exponential.
// Only the state carries a dependence from block to block (through Yoff and the epilogue); the
// mask and the products Y, S_acc of a block do not wait for the state. The math warps therefore
// run one block apart: mask block j, then (while the tensor core computes Y_j and S_acc_j) the
// epilogue of block j-1, then the scan of dt A for block j+1. Tensor memory holds G twice, M
// and Yoff; once a G buffer is masked, Y (columns 0-63) and S_acc (64-127) of that block are
// accumulated into it. Shared memory holds C and B twice and x three times, so that:
//   * G of block j+1 is computed while the math warps finish block j-1 and scan block j+1,
//   * Yoff of block j is computed as soon as the state S_{j-1} is written,
//   * C, B and x of later blocks are loaded while the current ones are worked on; the raw dt of
//     a block is copied two blocks ahead with cp.async, so no register waits on it.
// Hand-offs go through mbarriers (tcgen05.commit for the MMAs, TMA transaction counts for
// the loads, one elected arrival per phase of the math warps); every wait is bounded.
//
// Data layouts: TMA (4-D maps, 128-byte swizzle) brings C and B blocks (128 x 128) and x blocks
// (128 x 64) into shared memory in the canonical layouts the MMAs read directly (C and B
// K-major for G and Yoff; B as the MN-major A operand of the state product; x, w o x and the
// bf16 state MN-major as B operands). y is staged in the x buffer of its block.
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
constexpr int kMath = 256;       // 8 math warps
constexpr int kThreads = kMath + 32;   // + the control warp
constexpr uint32_t kTmemCols = 512;   // 384 used (a power of two is allocated)
constexpr uint32_t kColG = 0;    // G, two buffers of 128 columns; once masked, a buffer holds
                                 // Y (columns 0-63) and the state product (64-127) of its block
constexpr uint32_t kColM = 256;  // M in bf16 pairs (64 columns)
constexpr uint32_t kColYoff = 320;

constexpr int kAtom = 16384;     // 128 rows x 128 bytes
constexpr int kSmC = 0;                       // C, 2 stages x 2 atoms
constexpr int kSmB = kSmC + 4 * kAtom;        // B, 2 stages x 2 atoms
constexpr int kSmXw = kSmB + 4 * kAtom;       // w o x, 1 atom
constexpr int kSmX = kSmXw + kAtom;           // x (then y), 3 stages
constexpr int kSmS = kSmX + 3 * kAtom;        // bf16 state
constexpr int kSmDl = kSmS + kAtom;           // raw delta words, 2 buffers x kQ x 4 bytes
constexpr int kSmArr = kSmDl + 2 * kQ * 4;    // per block (2 buffers): cs, dt, e, w, v, each float[kQ]
constexpr int kNArr = 5;
constexpr int kSmRed = kSmArr + 2 * kNArr * kQ * 4;   // float[8]
constexpr int kNumBars = 11;
constexpr int kSmBar = kSmRed + 64;           // kNumBars mbarriers
constexpr int kSmTmem = kSmBar + kNumBars * 8;
constexpr int kSmFlag = kSmTmem + 8;
constexpr int kSmemUsed = kSmFlag + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024 bytes

constexpr uint32_t kIdescG = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescYoff = tc::idesc_bf16(128, 64, false, true);
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

// 4-byte asynchronous global -> shared copy (no register is tied up while it is in flight).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 r;
    r.x = tc::pack_bf16(v[0], v[1]);
    r.y = tc::pack_bf16(v[2], v[3]);
    r.z = tc::pack_bf16(v[4], v[5]);
    r.w = tc::pack_bf16(v[6], v[7]);
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
ssd_tc_kernel(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mB,
              const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap mY, const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
    float* red = reinterpret_cast<float*>(sm + kSmRed);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSmBar);
    uint64_t* full_cb = bars + 0;      // [2] C and B of a stage loaded
    uint64_t* full_x = bars + 2;       // [3] x of a stage loaded
    uint64_t* g_done = bars + 5;       // [2] G of a buffer computed
    uint64_t* yoff_done = bars + 7;    // Yoff of the block computed (all earlier MMAs too)
    uint64_t* mma2_done = bars + 8;    // Y and the state product computed
    uint64_t* math_ready = bars + 9;   // M and w o X of the block written, G read
    uint64_t* epi_done = bars + 10;    // state and y of the block written, accumulators read
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kSmTmem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmFlag);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;
    const int grp = h / p.heads_per_group;
    const int64_t L = p.seqlen;
    const int H = p.nheads;
    const int nblk = p.nblocks;

    if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (tid == kMath) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&mX);
        prefetch_tensormap(&mB);
        prefetch_tensormap(&mC);
        prefetch_tensormap(&mY);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == kMath / 32) {
        // ============================ control warp (one lane) ============================
        if (lane == 0) {
            const uint32_t aS = smem_u32(sm + kSmS), aXw = smem_u32(sm + kSmXw);
            auto aC = [&](int s) { return smem_u32(sm + kSmC + s * 2 * kAtom); };
            auto aB = [&](int s) { return smem_u32(sm + kSmB + s * 2 * kAtom); };
            auto aX = [&](int j) { return smem_u32(sm + kSmX + (j % 3) * kAtom); };
            auto load_cb = [&](int j) {
                const int s = j & 1;
                mbar_arrive_expect_tx(&full_cb[s], 4 * kAtom);
                tma_load_4d(sm + kSmC + s * 2 * kAtom, &mC, 0, grp, j * kQ, b, &full_cb[s]);
                tma_load_4d(sm + kSmC + s * 2 * kAtom + kAtom, &mC, 64, grp, j * kQ, b, &full_cb[s]);
                tma_load_4d(sm + kSmB + s * 2 * kAtom, &mB, 0, grp, j * kQ, b, &full_cb[s]);
                tma_load_4d(sm + kSmB + s * 2 * kAtom + kAtom, &mB, 64, grp, j * kQ, b, &full_cb[s]);
            };
            auto load_x = [&](int j) {
                const int s = j % 3;
                mbar_arrive_expect_tx(&full_x[s], kAtom);
                tma_load_4d(sm + kSmX + s * kAtom, &mX, 0, h, j * kQ, b, &full_x[s]);
            };
            auto issue_g = [&](int j) {
                const int s = j & 1;
#pragma unroll
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t off = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_ss(tmem + kColG + 128 * s, tc::sdesc_sw128(aC(s) + off, 16, 1024),
                               tc::sdesc_sw128(aB(s) + off, 16, 1024), kIdescG, k > 0);
                }
                tc::commit(&g_done[s]);
            };
            bool ok = true;
            auto wait = [&](uint64_t* bar, unsigned parity) {
                if (ok && !mbar_wait_bounded(bar, parity, p.status)) ok = false;
                return ok;
            };
            if (nblk > 0) {
                load_cb(0);
                load_x(0);
                if (nblk > 1) {
                    load_cb(1);
                    load_x(1);
                }
                if (nblk > 2) load_x(2);
                if (wait(&full_cb[0], 0)) {
                    tc::fence_after_sync();
                    issue_g(0);
                }
            }
            for (int j = 0; j < nblk && ok; ++j) {
                const int s = j & 1;
                // Y_j = M_j X_j and S_acc_j = B_j^T (w o X_j), into the columns of G_j, once
                // the math warps have masked G_j and written M_j and w o X_j
                if (!wait(math_ready, j & 1) || !wait(&full_x[j % 3], (j / 3) & 1)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    tc::mma_ts(tmem + kColG + 128 * s, tmem + kColM + 8 * k,
                               tc::sdesc_sw128(aX(j) + k * 2048, kAtom, 1024), kIdescY, k > 0);
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    tc::mma_ss(tmem + kColG + 128 * s + 64, tc::sdesc_sw128(aB(s) + k * 2048, kAtom, 1024),
                               tc::sdesc_sw128(aXw + k * 2048, kAtom, 1024), kIdescS, k > 0);
                tc::commit(mma2_done);
                // the state S_{j-1} is written and the accumulators of block j-1 are read
                if (!wait(epi_done, j & 1)) break;
                tc::fence_after_sync();
                if (j > 0) {
                    // y of block j-1 (staged in its x buffer) leaves
                    tma_store_4d(&mY, 0, h, (j - 1) * kQ, b, sm + kSmX + ((j - 1) % 3) * kAtom);
                    tma_store_commit();
                }
                // G_{j+1} into the buffer block j-1's accumulators have left
                if (j + 1 < nblk) {
                    if (!wait(&full_cb[s ^ 1], ((j + 1) >> 1) & 1)) break;
                    tc::fence_after_sync();
                    issue_g(j + 1);
                }
                // Yoff_j = C_j S_{j-1}
#pragma unroll
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t off = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_ss(tmem + kColYoff, tc::sdesc_sw128(aC(s) + off, 16, 1024),
                               tc::sdesc_sw128(aS + k * 2048, kAtom, 1024), kIdescYoff, k > 0);
                }
                tc::commit(yoff_done);
                // x_{j+2} takes the buffer of y_{j-1} once the store has read it
                if (j > 0 && j + 2 < nblk) {
                    tma_store_wait_read<0>();
                    load_x(j + 2);
                }
                // C_j and B_j are free once Yoff_j (and everything before it) is done
                if (j + 2 < nblk) {
                    if (!wait(yoff_done, j & 1)) break;
                    load_cb(j + 2);
                }
            }
            if (ok && nblk > 0) {
                // the last y
                if (wait(epi_done, nblk & 1)) {
                    tma_store_4d(&mY, 0, h, (nblk - 1) * kQ, b, sm + kSmX + ((nblk - 1) % 3) * kAtom);
                    tma_store_commit();
                }
            }
            tma_store_wait_all();
            if (!ok) *abort_flag = 1;
        }
    } else {
        // ============================ math warps ============================
        const int quarter = warp & 3;        // the TMEM lanes (rows) this warp can access
        const int half = warp >> 2;          // which half of the columns (or atom) it takes
        const int row = tid & 127;           // = 32 quarter + lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        const float Ah = p.A[h];
        const float bias = p.bias ? p.bias[h] : 0.f;
        const float Dh = p.D ? p.D[h] : 0.f;
        const __nv_bfloat16* delta = static_cast<const __nv_bfloat16*>(p.delta);
        auto arr = [&](int buf, int which) {
            return reinterpret_cast<float*>(sm + kSmArr) + (buf * kNArr + which) * kQ;
        };
        // a bounded wait whose outcome is the same for the whole warp (the warp-collective
        // tensor-memory accesses that follow must be taken by all its lanes or none)
        auto wait_warp = [&](uint64_t* bar, unsigned parity) {
            const bool okl = mbar_wait_bounded(bar, parity, p.status);
            return __all_sync(0xffffffffu, okl) != 0;
        };
        // all math threads done with a phase: one arrival; false if any thread failed
        auto signal = [&](uint64_t* bar, bool okt) -> bool {
            const bool bad = named_bar_or(1, kMath, !okt || *abort_flag);
            if (tid == 0) mbar_arrive(bar);
            return !bad;
        };
        // raw delta of block j, row `row`: the aligned 4-byte word holding it is copied into
        // shared memory (buffer j & 1) without tying up a register; one commit group per block
        const uintptr_t dl_hi = 2;
        auto load_delta = [&](int j) {
            const int64_t tt = (int64_t)j * kQ + row;
            if (half == 0 && j < nblk && tt < L &&
                idx_ok(((int64_t)b * L + tt) * H + h, (int64_t)gridDim.y * L * H, p.status)) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(delta + ((int64_t)b * L + tt) * H + h);
                cp_async4(sm + kSmDl + (j & 1) * kQ * 4 + row * 4, reinterpret_cast<const void*>(a & ~(uintptr_t)3));
            }
            cp_async_commit();
        };
        auto read_delta = [&](int j) -> float {
            const int64_t tt = (int64_t)j * kQ + row;
            if (half != 0 || tt >= L) return 0.f;
            const uintptr_t a = reinterpret_cast<uintptr_t>(delta + ((int64_t)b * L + tt) * H + h);
            const uint32_t w = *reinterpret_cast<const uint32_t*>(sm + kSmDl + (j & 1) * kQ * 4 + row * 4);
            return (a & dl_hi) ? bf_hi(w) : bf_lo(w);
        };
        // the block scan of dt A_h for block j into array buffer j & 1 (first warpgroup)
        auto scan_block = [&](int j, float draw) {
            const int buf = j & 1;
            float dt = 0.f, cum = 0.f;
            if (half == 0) {
                if ((int64_t)j * kQ + row < L) {
                    const float v = draw + bias;
                    dt = p.softplus ? softplus_accurate(v) : v;
                }
                cum = dt * Ah;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, cum, o);
                    if (lane >= o) cum += n;
                }
                if (lane == 31) red[warp] = cum;
            }
            named_bar_or(1, kMath, false);
            if (half == 0) {
                float before = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    if (w < warp) before += red[w];
                cum += before;
                const float cum_last = red[0] + red[1] + red[2] + red[3];
                const float cs_t = cum * kLog2e;
                arr(buf, 0)[row] = cs_t;
                arr(buf, 1)[row] = dt;
                arr(buf, 2)[row] = ex2_approx(cs_t);
                arr(buf, 3)[row] = ex2_approx((cum_last - cum) * kLog2e) * dt;
                // v_s = dt_s exp(cum_ref - cum_s), cum_ref the cumulative sum at the last step of
                // the 32-step chunk of s (this warp's lane 31): cum_ref <= cum_s, so v_s <= dt_s
                const float cs_ref = __shfl_sync(0xffffffffu, cs_t, 31);
                arr(buf, 4)[row] = dt * ex2_approx(cs_ref - cs_t);
                if (row == 0) red[4 + buf] = ex2_approx(cum_last * kLog2e);
            }
            named_bar_or(1, kMath, false);
        };

        // initial state: row `row`, columns [32 half, +32) in registers, bf16 copy in sS
        float S[kP / 2];
        {
            const int64_t is = (((int64_t)b * H + h) * kN + row) * kP + 32 * half;
            const float* src =
                p.h0 && idx_ok(is + 31, (int64_t)gridDim.y * H * kN * kP, p.status) ? p.h0 + is : nullptr;
#pragma unroll
            for (int i = 0; i < kP / 2; i += 4) {
                const float4 v = src ? *reinterpret_cast<const float4*>(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[i] = v.x;
                S[i + 1] = v.y;
                S[i + 2] = v.z;
                S[i + 3] = v.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(sm + kSmS + sw128(row, 4 * half + c)) = pack8(S + 8 * c);
        }
        load_delta(0);
        load_delta(1);
        cp_async_wait<1>();
        scan_block(0, read_delta(0));
        fence_proxy_async_smem();
        bool ok = signal(epi_done, true);    // the initial state is in place

        // epilogue of block jj: y rows into x buffer jj % 3, the state row. Inside the loop the
        // products of block jj were waited for at the top of block jj + 1 (by then those of
        // jj + 1 may be done as well, and a second parity wait would take their phase for it)
        auto epilogue = [&](int jj, bool wait_mma2) -> bool {
            const int sj = jj & 1;
            bool okw = !wait_mma2 || wait_warp(mma2_done, jj & 1);
            okw = okw && wait_warp(yoff_done, jj & 1);
            tc::fence_after_sync();
            if (okw) {
                const int64_t t = (int64_t)jj * kQ + row;
                const float e_t = arr(sj, 2)[row];
                const float e_last = red[4 + sj];
                const int64_t irow = (((int64_t)b * L + t) * H + h) * kP + 32 * half;
                const bool row_ok = t < L && idx_ok(irow + 31, (int64_t)gridDim.y * L * H * kP, p.status);
                const __nv_bfloat16* xrow = p.D && row_ok ? static_cast<const __nv_bfloat16*>(p.x) +
                                                               (((int64_t)b * L + t) * H + h) * kP + 32 * half
                                                         : nullptr;
                const __nv_bfloat16* zrow = p.z && row_ok ? static_cast<const __nv_bfloat16*>(p.z) +
                                                               (((int64_t)b * L + t) * H + h) * kP + 32 * half
                                                         : nullptr;
                unsigned char* ys = sm + kSmX + (jj % 3) * kAtom;
                const uint32_t colY = kColG + 128 * sj;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t ry[16], ro[16];
                    tc::ld16(lane_base + colY + 32 * half + 16 * q, ry);
                    tc::ld16(lane_base + kColYoff + 32 * half + 16 * q, ro);
                    tc::wait_ld();
                    float yv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) yv[i] = fmaf(e_t, __uint_as_float(ro[i]), __uint_as_float(ry[i]));
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
                    for (int c = 0; c < 2; ++c)
                        *reinterpret_cast<uint4*>(ys + sw128(row, 4 * half + 2 * q + c)) = pack8(yv + 8 * c);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t rs[16];
                    tc::ld16(lane_base + colY + 64 + 32 * half + 16 * q, rs);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) S[16 * q + i] = fmaf(e_last, S[16 * q + i], __uint_as_float(rs[i]));
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        *reinterpret_cast<uint4*>(sm + kSmS + sw128(row, 4 * half + 2 * q + c)) =
                            pack8(S + 16 * q + 8 * c);
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            return signal(epi_done, okw);
        };

        for (int j = 0; j < nblk && ok; ++j) {
            const int s = j & 1;
            const float* cs = arr(s, 0);
            const float* dts = arr(s, 1);
            const float* vs = arr(s, 4);
            // delta of block j+2 (block j's buffer: its scan is done)
            load_delta(j + 2);
            // ---- wait for x_j and G_j, and for block j-1's products to have consumed M and w o X
            bool okw = wait_warp(&full_x[j % 3], (j / 3) & 1) && wait_warp(&g_done[s], (j >> 1) & 1);
            if (okw && j > 0) okw = wait_warp(mma2_done, (j - 1) & 1);
            tc::fence_after_sync();
            if (okw) {
                // ---- mask: M[t, s'] = G[t, s'] exp(cum_t - cum_s') dt_s' for s' <= t. Warp
                // (quarter, half) takes the 16-column half `half` of each 32-column chunk kc of
                // its rows: below the diagonal chunk (kc < quarter) a factored decay, on it one
                // exponential per element, above it zeros; both warps of a quarter get the same
                // mix of work
                const float cs_t = cs[row];
#pragma unroll
                for (int kc = 0; kc < 4; ++kc) {
                    const int c0 = 32 * kc + 16 * half;   // first column of this half-chunk
                    uint32_t packed[8];
                    if (kc <= quarter) {
                        uint32_t r[16];
                        tc::ld16(lane_base + kColG + 128 * s + c0, r);
                        tc::wait_ld();
                        if (kc < quarter) {
                            // below the diagonal: exp(cum_t - cum_s) dt_s = f_t v_s with
                            // f_t = exp(cum_t - cum_ref) <= 1 (t is past the chunk)
                            const float f = ex2_approx(cs_t - cs[32 * kc + 31]);
                            const f2 f2v = pk(f, f);
#pragma unroll
                            for (int i = 0; i < 16; i += 4) {
                                const ulonglong2 v4 = *reinterpret_cast<const ulonglong2*>(vs + c0 + i);
                                float m0, m1, m2, m3;
                                upk(mul2(mul2(pk(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), v4.x), f2v), m0, m1);
                                upk(mul2(mul2(pk(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])), v4.y), f2v), m2,
                                    m3);
                                packed[i / 2] = tc::pack_bf16(m0, m1);
                                packed[i / 2 + 1] = tc::pack_bf16(m2, m3);
                            }
                        } else {
                            // the diagonal chunk: s <= t, exp(cum_t - cum_s) directly
                            const int lim = lane - 16 * half;   // columns i <= lim are at or below t
#pragma unroll
                            for (int i = 0; i < 16; i += 4) {
                                const float4 c4 = *reinterpret_cast<const float4*>(cs + c0 + i);
                                const float4 d4 = *reinterpret_cast<const float4*>(dts + c0 + i);
                                const float m0 = i <= lim ? __uint_as_float(r[i]) * d4.x * ex2_approx(cs_t - c4.x) : 0.f;
                                const float m1 =
                                    i + 1 <= lim ? __uint_as_float(r[i + 1]) * d4.y * ex2_approx(cs_t - c4.y) : 0.f;
                                const float m2 =
                                    i + 2 <= lim ? __uint_as_float(r[i + 2]) * d4.z * ex2_approx(cs_t - c4.z) : 0.f;
                                const float m3 =
                                    i + 3 <= lim ? __uint_as_float(r[i + 3]) * d4.w * ex2_approx(cs_t - c4.w) : 0.f;
                                packed[i / 2] = tc::pack_bf16(m0, m1);
                                packed[i / 2 + 1] = tc::pack_bf16(m2, m3);
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) packed[i] = 0u;
                    }
                    tc::st8(lane_base + kColM + c0 / 2, packed);
                }
                // ---- w o X_j: thread tid takes row tid / 2, chunks 4 (tid & 1) .. + 3, walked so
                // that the eight lanes of a shared-memory phase hit eight bank groups
                {
                    const int xr = tid >> 1, xg = tid & 1;
                    const float wt = arr(s, 3)[xr];
                    const f2 w2 = pk(wt, wt);
                    const unsigned char* src = sm + kSmX + (j % 3) * kAtom + xr * 128;
                    unsigned char* dst = sm + kSmXw + xr * 128;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = (4 * xg + i) ^ (xr & 7);
                        *reinterpret_cast<uint4*>(dst + 16 * c) =
                            scale_bf16x8(*reinterpret_cast<const uint4*>(src + 16 * c), w2);
                    }
                }
                tc::wait_st();
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            ok = signal(math_ready, okw);
            if (!ok) break;

            // ---- the epilogue of the previous block while the tensor core works on this one
            if (j > 0) {
                ok = epilogue(j - 1, false);
                if (!ok) break;
            }

            // ---- the scan of the next block
            cp_async_wait<1>();
            if (j + 1 < nblk) scan_block(j + 1, read_delta(j + 1));
        }
        if (ok && nblk > 0) ok = epilogue(nblk - 1, true);
        cp_async_wait<0>();   // no copy may land after the block has left
        if (ok && p.h_last &&
            idx_ok((((int64_t)b * H + h) * kN + row) * kP + 32 * half + 31, (int64_t)gridDim.y * H * kN * kP,
                   p.status)) {
            float* dst = p.h_last + (((int64_t)b * H + h) * kN + row) * kP + 32 * half;
#pragma unroll
            for (int i = 0; i < kP / 2; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
        }
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
    p.status = a.status;
    if (!p.status) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once<ssd_tc_kernel>(kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.nheads, (unsigned)a.batch);
    ssd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mX, mB, mC, mY, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
