// Instantiations of the time-parallel chunk scan (scan_tp_kernel.cuh): 2 or 4
// time lanes per channel, fp32 or bf16 inputs.
#include "scan_tp_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_tp(int dtype, int time_lanes, const ScanArgs& a, const ScanMaps& maps, dim3 grid,
                           cudaStream_t stream) {
  if (dtype == 0) {
    if (time_lanes == 2) return launch_scan_tp_variant<float, 2>(a, maps, grid, stream);
    if (time_lanes == 4) return launch_scan_tp_variant<float, 4>(a, maps, grid, stream);
  } else {
    if (time_lanes == 2) return launch_scan_tp_variant<__nv_bfloat16, 2>(a, maps, grid, stream);
    if (time_lanes == 4) return launch_scan_tp_variant<__nv_bfloat16, 4>(a, maps, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mamba
