// Instantiations of the backward kernel's two segment passes: the forward
// aggregate (segments 0..S-2) and the adjoint aggregate (segments 1..S-1).
#include "scan_bwd_kernel.cuh"

namespace mamba {

cudaError_t launch_scan_bwd_fwd_agg(int dtype, const BwdArgs& a, cudaStream_t stream) {
  return launch_bwd_mode<kBwdFwdAgg>(dtype, a, unsigned(a.nseg - 1), stream);
}

cudaError_t launch_scan_bwd_adj_agg(int dtype, const BwdArgs& a, cudaStream_t stream) {
  return launch_bwd_mode<kBwdAdjAgg>(dtype, a, unsigned(a.nseg - 1), stream);
}

}  // namespace mamba
