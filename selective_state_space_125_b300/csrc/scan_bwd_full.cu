// Instantiations of the backward kernel's full pass (the gradients).
#include "scan_bwd_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_bwd_full(int dtype, const BwdArgs& a, cudaStream_t stream) {
  return launch_bwd_mode<kBwdFull>(dtype, a, unsigned(a.nseg), stream);
}

}  // namespace mamba
