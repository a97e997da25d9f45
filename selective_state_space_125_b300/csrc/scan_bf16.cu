// bf16-input, zero-order-hold instantiations of the scan kernels.
#include "scan_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_bf16_d0(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps,
                                dim3 grid, cudaStream_t stream) {
  return launch_scan_typed<__nv_bfloat16, 0>(npl, lpc, mode, a, maps, grid, stream);
}

bool scan_variant_bf16(int npl, int lpc, ScanVariant* v) { return scan_variant_typed<__nv_bfloat16>(npl, lpc, v); }

}  // namespace mamba
