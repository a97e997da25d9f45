// fp32-input instantiations of the scan kernels (precise math path).
#include "scan_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_f32(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps, dim3 grid,
                            cudaStream_t stream) {
  return launch_scan_typed<float>(npl, lpc, mode, a, maps, grid, stream);
}

bool scan_variant_f32(int npl, int lpc, ScanVariant* v) { return scan_variant_typed<float>(npl, lpc, v); }

}  // namespace mamba
