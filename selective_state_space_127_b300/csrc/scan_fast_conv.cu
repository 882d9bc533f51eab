// The fast selective-scan kernels with the causal conv1d + SiLU prologue on x, instantiated in
// a translation unit of their own (see scan_fast.cuh and the notes at the top of scan_fast.cu).
#include "scan_fast.cuh"

namespace ssm {
namespace fast {

cudaError_t dispatch_conv_full(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                               cudaStream_t st) {
    return dispatch<kFull, kVarConv>(maps, fp, a, nz, st);
}

cudaError_t dispatch_conv_pass1(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                                cudaStream_t st) {
    return dispatch<kPass1, kVarConv>(maps, fp, a, nz, st);
}

}  // namespace fast
}  // namespace ssm
