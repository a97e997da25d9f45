// fp32-input zero-order-hold scan kernels with the causal conv1d + SiLU fused in front.
#include "scan_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_f32_conv(int npl, int lpc, ScanMode mode, const ScanArgs& a, const ScanMaps& maps,
                                 dim3 grid, cudaStream_t stream) {
  return launch_scan_typed<float, 0, true>(npl, lpc, mode, a, maps, grid, stream);
}

}  // namespace mamba
