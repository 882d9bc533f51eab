// Internal interface between the C-ABI layer (api.cu) and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "ssmscan.h"

namespace ssm {

// Host-validated selective-scan arguments, passed to kernels by value.
struct ScanArgs {
    int64_t batch, seqlen, dim;
    int dstate;
    int io_bf16;
    int softplus, reverse, zoh;
    const void* x;
    const void* delta;
    const void* B;
    const void* C;
    const void* z;
    const float* A;
    const float* D;
    const float* bias;
    const float* h0;
    void* y;
    float* h_last;
    int64_t xs[3], ds[3], zs[3], ys[3], Bs[3], Cs[3];
    int64_t chunk_len;
    void* workspace;
    size_t workspace_bytes;
    int debug_flags;
    int algorithm;           // SSM_SCAN_ALGO_SERIAL or SSM_SCAN_ALGO_ASSOC
    // causal conv1d + SiLU prologue on x (conv_w == nullptr: none)
    const float* conv_w;     // (D, K)
    const float* conv_b;     // (D) or nullptr
    const void* conv_prev;   // (b, K-1, D) io dtype or nullptr
    int conv_k;
    unsigned* status;        // the workspace header's status word (nullptr when no workspace)
    void* const* phase_events;   // cudaEvent_t handles recorded around the launches, or nullptr
    int n_phase_events;
    // element extents (largest index + 1) of the strided views x, delta, z, y, B, C: the bounds
    // the debug build checks computed indices against
    int64_t ext_x, ext_delta, ext_z, ext_y, ext_B, ext_C;
};

struct Conv1dArgs {
    int64_t batch, seqlen, dim;
    int k;
    int io_bf16;
    int silu;
    const void* x;
    const float* w;
    const float* bias;
    const void* x_prev;
    void* y;
    unsigned* status;        // the workspace header's status word
};

struct SSDArgs {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
    int io_bf16;
    int softplus;
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* bias;
    const float* h0;
    void* y;
    float* h_last;
    void* workspace;
    size_t workspace_bytes;
    unsigned* status;        // the workspace header's status word (tensor-core path)
};

// Which selective-scan kernel a call takes.
enum class ScanPath { Generic = 0, Fast = 1, ChunkCarry = 2 };

// Opt kernel KERN into `bytes` (a constant per kernel) of dynamic shared memory above the
// default 48 KB, once per device: the attribute outlives the call, so later launches skip it.
template <auto KERN>
cudaError_t set_smem_once(int bytes) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Once per kernel and device: ask for the largest shared-memory carveout, so that as many CTAs
// as their shared memory allows can be resident (the default carveout leaves more L1 and fewer
// CTAs), and raise the dynamic shared-memory limit when `bytes` is above the default 48 KB.
template <auto KERN>
cudaError_t set_max_carveout_once(int bytes) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && bytes > 48 * 1024)
        e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Record a reason for ssm_last_error() on the calling thread; returns `s`.
ssm_status_t set_error(ssm_status_t s, const char* msg);

// Count of kernels enqueued by this library (reported through ssm_kernel_launch_count).
void note_launches(int n);

// Record the phase events of a call: before the first launch (k = 0) or after the k-th launch;
// after the last launch (last = true) every remaining event is recorded too.
cudaError_t record_phase(const ScanArgs& a, int k, bool last, cudaStream_t st);

// Device address of the status header of the built-in scratch of ssm_scan_fwd_noalloc on the
// current device (looked up on first use); nullptr with the CUDA error in *err on failure.
void* noalloc_scratch(cudaError_t* err);

// Kernel launchers: return cudaSuccess or the launch error. They assume valid args.
cudaError_t launch_conv1d(const Conv1dArgs& a, cudaStream_t st);
bool scan_decode_supported(const ScanArgs& a);
cudaError_t launch_scan_decode(const ScanArgs& a, cudaStream_t st);
cudaError_t launch_scan_generic(const ScanArgs& a, cudaStream_t s);
bool scan_fast_supported(const ScanArgs& a);
// Steps per chunk the fast path uses (a multiple of its tile; >= seqlen when not split) and
// the workspace bytes it needs after the header for the chunk carries (0 when the sequence
// is not split).
int64_t scan_fast_chunk(const ScanArgs& a);
size_t scan_fast_workspace_bytes(const ScanArgs& a);
cudaError_t launch_scan_fast(const ScanArgs& a, cudaStream_t s);
cudaError_t launch_ssd_reference(const SSDArgs& a, cudaStream_t s);
// Tensor-core SSD path: bf16 I/O, P = 64, N = 128, chunk a multiple of 128, TMA-aligned.
bool ssd_tc_supported(const SSDArgs& a);
cudaError_t launch_ssd_tc(const SSDArgs& a, cudaStream_t s);

}  // namespace ssm
