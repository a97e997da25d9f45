// fp32-input, simplified-Bbar instantiations of the scan kernels.
#include "scan_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_f32_d1(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps,
                                dim3 grid, cudaStream_t stream) {
  return launch_scan_typed<float, 1>(npl, lpc, mode, a, maps, grid, stream);
}

}  // namespace mamba
