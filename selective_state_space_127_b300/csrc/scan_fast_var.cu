// The fast selective-scan kernels of the exact zero-order-hold discretisation and of the reverse
// direction, instantiated in a translation unit of their own (see scan_fast.cuh and the notes at
// the top of scan_fast.cu).
#include "scan_fast.cuh"

namespace ssm {
namespace fast {

cudaError_t dispatch_zoh_full(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                              cudaStream_t st) {
    return dispatch<kFull, kVarZoh>(maps, fp, a, nz, st);
}

cudaError_t dispatch_zoh_pass1(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                               cudaStream_t st) {
    return dispatch<kPass1, kVarZoh>(maps, fp, a, nz, st);
}

cudaError_t dispatch_rev_full(const CUtensorMap* maps, const FastParams& fp, const ScanArgs& a, int nz,
                              cudaStream_t st) {
    return dispatch<kFull, kVarRev>(maps, fp, a, nz, st);
}

}  // namespace fast
}  // namespace ssm
