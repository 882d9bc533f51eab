// ssm_scan_fwd_noalloc: the selective scan for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a host application whose device
// memory is planned once at start-up and may not grow afterwards, a plugin running inside
// another runtime that owns every device allocation and passes only the tensors, or a
// latency-critical loop that cannot afford cudaMalloc (which may synchronise the device and
// can fail under memory pressure). For them this entry point takes the scratch of the
// chunked (long-sequence) scan from a fixed buffer compiled into the library instead of
// from a caller-provided workspace. Inputs and outputs are still the caller's.
//
// The buffer is a file-scope device array, so every GPU that loads the library holds it
// until the process exits. In host code its name does not denote a device address; the
// address is looked up once per device, with that device current, by cudaGetSymbolAddress,
// and only that address is handed to the kernels. Like any workspace it starts with the
// status header (zero when the module loads; ssm_check_status(NULL, ...) reads and clears it)
// followed by the chunk carries. All calls share the buffer and it keeps the contents of the
// last call; the carries need no zeroing, because the chunked scan writes every element it
// later reads. Calls whose work overlaps on the GPU race on it.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ssmscan.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

namespace ssm {

// Device address of g_noalloc_scratch on the current device (looked up on first use).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = addr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

void* noalloc_scratch(cudaError_t* err) {
    void* p = nullptr;
    *err = scratch_address(&p);
    return *err == cudaSuccess ? p : nullptr;
}

}  // namespace ssm

extern "C" ssm_status_t ssm_scan_fwd_noalloc(const ssm_scan_params* p, void* stream) {
    const size_t need = ssm_scan_workspace_size(p);
    if (need == (size_t)-1) return ssm_scan_fwd(p, stream);   // reports the argument error, launches nothing
    if (need > (size_t)SSM_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "this call needs %zu bytes of scratch; the built-in scratch of ssm_scan_fwd_noalloc holds %zu "
                 "(use ssm_scan_fwd with a workspace, or a larger chunk_len)",
                 need, (size_t)SSM_NOALLOC_SCRATCH_BYTES);
        return ssm::set_error(SSM_ERR_UNSUPPORTED, msg);
    }
    ssm_scan_params q = *p;
    q.workspace = nullptr;
    q.workspace_bytes = 0;
    if (need > 0) {
        void* scratch = nullptr;
        const cudaError_t e = ssm::scratch_address(&scratch);
        if (e != cudaSuccess) {
            char msg[200];
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch: %s", cudaGetErrorString(e));
            return ssm::set_error(SSM_ERR_CUDA, msg);
        }
        q.workspace = scratch;
        q.workspace_bytes = SSM_NOALLOC_SCRATCH_BYTES;
    }
    return ssm_scan_fwd(&q, stream);
}

extern "C" size_t ssm_noalloc_scratch_bytes(void) { return (size_t)SSM_NOALLOC_SCRATCH_BYTES; }
