// Fast selective-scan kernels for dense channel-contiguous layouts (the Mamba block's
// (b, L, D) activations and (b, L, N) B, C), N in {16, 32, 64}, delta*B discretisation, with
// an optional split of the sequence into chunks; variants (one per kernel) add the conv1d +
// SiLU prologue on x, the exact zero-order hold B_bar = (A_bar - 1) / A B (a series in
// z = dt A for |z| < 1/8, where the difference would cancel), or walk the sequence backwards
// (tiles in reverse order, rows of a tile from last to first; one chunk).
//
// Work split. A CTA owns kCh = 16 consecutive channels of one batch row and walks one
// chunk of the sequence (the whole sequence when it is not split). LPC lanes share a
// channel, lane g keeping the fp32 states n in [g S, g S + S), S = N / LPC, in registers.
//
// Data movement. TMA (3-D tensor maps over (D or N, L, b)) streams 32-step tiles of x,
// delta, z, B and C into a 2-deep shared-memory ring guarded by mbarriers; y tiles leave
// through TMA stores from one staging tile (the store of a tile has long finished reading it
// when the next tile's outputs are written). B and C tiles are widened to fp32 once per tile
// by the CTA, so lanes then read their states' values with 8- or 16-byte loads. The local pass
// loads neither z nor C and stages no y, so its CTAs take about half the shared memory.
//
// Steps go in supergroups of 2 LPC. Lane g of a channel computes the per-(t, channel) scalars
// of steps g and g + LPC of the supergroup (dt = softplus(delta + bias), dt x, silu(z), D x)
// as packed pairs (f32x2 arithmetic, a branch-free softplus) one supergroup ahead, so that
// chain overlaps the state updates of the current supergroup; the (dt, dt x) values are then
// broadcast inside the channel's lanes. Per step and state:
//   A_bar[n] = 2^(dt * A[n] * log2 e)           SFU ex2
//   h[n] = A_bar[n] h[n] + (dt x) B[n]          packed fp32 pairs (fma.rn.f32x2)
//   y += C[n] h[n]                               packed pairs
// and the lanes' partial sums of each half of the supergroup are reduce-scattered (log2 LPC
// shuffle rounds), leaving lane g with the y of steps g and g + LPC, which it finishes as
// (y + D x) silu(z) on the pair.
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
// Conv prologue (CONV kernels): the x box of a tile starts kHalo = 3 rows early (zero-filled
// before t = 0, or the caller's previous inputs for the first tile), and the lane that forms a
// step's scalars first forms x_t = silu(bias + sum_j w[j] x_{t-3+j}) from those rows.
//
// Recurrence: "Mamba/SSM complete guide" section 5 `selective_scan` and MambaBlock.forward;
// "論文解説: Mamba" "選択機構" (softplus) and "Hardware-Aware Parallel Scan" (state kept
// on chip, only the outputs written back; the parallel scan over (A_bar, B_bar x) pairs).
#include <mutex>

#include "scan_fast.cuh"

namespace ssm {
using namespace fast;
namespace {

// Chunk carry: one thread per (b, d, n) walks the chunks in order,
//   H_0 = h0,  H_{c+1} = exp(A[d, n] * sumdt_c) * H_c + local_c,
// where slot c + 1 holds local_c (pass 1), and stores H_c into slot c: the initial state of
// every chunk, chunk 0's being a copy of h0 (so that h0 may alias h_last).
__global__ void scan_carry_kernel(float* carry, const float* sumdt, const float* A, const float* h0,
                                  int64_t batch, int64_t dim, int N, int nsteps, unsigned* status) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = batch * dim * N;
    if (i >= total) return;
    const int64_t bd = i / N;
    const int n = (int)(i % N);
    const int64_t d = bd % dim;
    const float a = idx_ok(d * N + n, dim * N, status) ? A[d * N + n] : 0.f;
    float H = h0 ? h0[i] : 0.f;
    carry[i] = H;
    // the local states and sums of eight chunks are loaded before any of them is combined, so
    // eight loads are in flight instead of one (each slot is read before this thread, its only
    // user, overwrites it)
    constexpr int kAhead = 8;
    for (int c0 = 0; c0 < nsteps; c0 += kAhead) {
        float loc[kAhead], sd[kAhead];
        bool ok = true;
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            const int c = c0 + j;
            loc[j] = 0.f;
            sd[j] = 0.f;
            if (c < nsteps) {
                const int64_t o = (int64_t)(c + 1) * total + i;
                const int64_t os = (int64_t)c * batch * dim + bd;
                if (idx_ok(o, (int64_t)(nsteps + 1) * total, status) &&
                    idx_ok(os, (int64_t)nsteps * batch * dim, status)) {
                    loc[j] = carry[o];
                    sd[j] = sumdt[os];
                } else {
                    ok = false;
                }
            }
        }
        if (!ok) break;
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            const int c = c0 + j;
            if (c < nsteps) {
                H = fmaf(expf(a * sd[j]), H, loc[j]);
                carry[(int64_t)(c + 1) * total + i] = H;
            }
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

// 3-D map over (inner, L, b) with element strides (1, st, sb) and box (box0, rows, 1).
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t L, int64_t b, int64_t st,
              int64_t sb, int box0, int rows = kT) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)b};
    const int64_t bstride = b > 1 ? sb * esz : ((L * st * esz + 15) / 16) * 16;
    cuuint64_t strides[2] = {(cuuint64_t)(st * esz), (cuuint64_t)bstride};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                    const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr int64_t kMinChunk = 512;    // shortest chunk the automatic split uses
constexpr int64_t kMaxChunks = 65535; // the grid's z extent

}  // namespace

bool scan_fast_supported(const ScanArgs& a) {
    const int N = a.dstate;
    if (N != 16 && N != 32 && N != 64) return false;
    // one variant per kernel: the conv prologue, exact ZOH or the reverse direction
    if ((a.conv_w != nullptr) + a.zoh + a.reverse > 1) return false;
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
    if (a.reverse) return ((L + kT - 1) / kT) * kT;   // the reverse kernel walks one chunk
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
    // at most kMaxChunks chunks: the chunk index is the grid's z dimension
    const int64_t min_q = (L + kMaxChunks - 1) / kMaxChunks;
    if (q < min_q) q = min_q;
    q = ((q + kT - 1) / kT) * kT;
    if (q >= L) q = ((L + kT - 1) / kT) * kT;
    return q;
}

size_t scan_fast_workspace_bytes(const ScanArgs& a) {
    if (a.seqlen == 0) return 0;
    const int64_t q = scan_fast_chunk(a);
    const int64_t nch = (a.seqlen + q - 1) / q;
    if (nch <= 1) return 0;
    return (size_t)(nch * a.batch * a.dim * a.dstate + (nch - 1) * a.batch * a.dim) * sizeof(float);
}

cudaError_t launch_scan_fast(const ScanArgs& a, cudaStream_t st) {
    CUtensorMap maps[6];
    const bool bf = a.io_bf16 != 0;
    const void* zsrc = a.z ? a.z : a.x;                 // unused map when there is no gate
    const int64_t* zst = a.z ? a.zs : a.xs;
    const bool conv = a.conv_w != nullptr;
    const bool assoc = a.algorithm == SSM_SCAN_ALGO_ASSOC;
    if (!make_map(&maps[0], a.x, bf, a.dim, a.seqlen, a.batch, a.xs[1], a.xs[0], kCh, conv ? kT + kHalo : kT) ||
        !make_map(&maps[1], a.delta, bf, a.dim, a.seqlen, a.batch, a.ds[1], a.ds[0], kCh) ||
        !make_map(&maps[2], zsrc, bf, a.dim, a.seqlen, a.batch, zst[1], zst[0], kCh) ||
        !make_map(&maps[3], a.B, bf, a.dstate, a.seqlen, a.batch, a.Bs[1], a.Bs[0], a.dstate) ||
        !make_map(&maps[4], a.C, bf, a.dstate, a.seqlen, a.batch, a.Cs[1], a.Cs[0], a.dstate) ||
        !make_map(&maps[5], a.y, bf, a.dim, a.seqlen, a.batch, a.ys[1], a.ys[0], kCh))
        return cudaErrorInvalidValue;
    const int64_t q = scan_fast_chunk(a);
    const int nch = (int)((a.seqlen + q - 1) / q);
    FastParams fp{a.seqlen, q, (int)a.dim, nch, a.A, a.D, a.bias, a.h0, a.h_last, nullptr, nullptr,
                  a.status, (a.debug_flags & SSM_DEBUG_SKIP_FIRST_LOAD) ? 1 : 0,
                  a.conv_w, a.conv_b, a.conv_prev, a.conv_k};
    if (!fp.status) return cudaErrorInvalidValue;
    cudaError_t e = record_phase(a, 0, false, st);
    if (e != cudaSuccess) return e;
    if (nch > 1) {
        // the carries follow the workspace header
        const size_t slot_floats = (size_t)(a.batch * a.dim * a.dstate);
        fp.carry = reinterpret_cast<float*>(static_cast<unsigned char*>(a.workspace) + SSM_WORKSPACE_HEADER_BYTES);
        fp.sumdt = fp.carry + (size_t)nch * slot_floats;
        e = assoc    ? dispatch_assoc_pass1(maps, fp, a, nch - 1, st)
            : conv   ? dispatch_conv_pass1(maps, fp, a, nch - 1, st)
            : a.zoh  ? dispatch_zoh_pass1(maps, fp, a, nch - 1, st)
                     : dispatch<kPass1, kVarPlain>(maps, fp, a, nch - 1, st);
        if (e == cudaSuccess) e = record_phase(a, 1, false, st);
        if (e != cudaSuccess) return e;
        const int64_t total = a.batch * a.dim * a.dstate;
        scan_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(fp.carry, fp.sumdt, a.A, a.h0, a.batch,
                                                                          a.dim, a.dstate, nch - 1, a.status);
        note_launches(1);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = record_phase(a, 2, false, st);
        if (e != cudaSuccess) return e;
    }
    e = assoc    ? dispatch_assoc_full(maps, fp, a, nch, st)
        : conv   ? dispatch_conv_full(maps, fp, a, nch, st)
        : a.zoh ? dispatch_zoh_full(maps, fp, a, nch, st)
        : a.reverse ? dispatch_rev_full(maps, fp, a, nch, st)
                    : dispatch<kFull, kVarPlain>(maps, fp, a, nch, st);
    if (e != cudaSuccess) return e;
    return record_phase(a, nch > 1 ? 3 : 1, true, st);
}

}  // namespace ssm
