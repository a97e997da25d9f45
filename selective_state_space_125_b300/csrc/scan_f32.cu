// fp32-input, zero-order-hold instantiations of the scan kernels.
#include "scan_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_f32_d0(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps,
                                dim3 grid, cudaStream_t stream) {
  return launch_scan_typed<float, 0>(npl, lpc, mode, a, maps, grid, stream);
}

bool scan_variant_f32(int npl, int lpc, ScanVariant* v) { return scan_variant_typed<float>(npl, lpc, v); }

}  // namespace mamba
