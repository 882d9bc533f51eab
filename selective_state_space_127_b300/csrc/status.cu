// The library's device status word (one per device): kernels whose bounded waits give up
// latch a nonzero ssm_status_t here; ssm_device_status() reads and optionally clears it.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace ssm {

__device__ unsigned int g_device_status = 0;

namespace {
constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;
}  // namespace

unsigned* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_status_ptr[dev];
}

cudaError_t read_device_status(unsigned* out, bool clear, cudaStream_t st) {
    unsigned* p = device_status_ptr();
    if (!p) return cudaErrorInvalidDevice;
    cudaError_t e = cudaMemcpyAsync(out, p, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(p, 0, sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

}  // namespace ssm
