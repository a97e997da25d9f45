// Backward of the selective scan: one call runs the segment passes (when the
// sequence is cut into segments) and the full pass, all on the call's stream.
// The kernels are in scan_bwd_kernel.cuh.
#include "bwd_args.h"

namespace mamba {

bool scan_bwd_supported(int dstate) { return dstate == 16 || dstate == 32 || dstate == 64 || dstate == 128; }

cudaError_t launch_scan_bwd(int dtype, const BwdArgs& a, cudaStream_t stream) {
  if (a.nseg > 1) {
    cudaError_t e = launch_scan_bwd_fwd_agg(dtype, a, stream);
    if (e == cudaSuccess) e = launch_scan_bwd_adj_agg(dtype, a, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_scan_bwd_full(dtype, a, stream);
}

}  // namespace mamba
