// Argument block and launcher of the single-token state update, shared by
// api.cu and state_update.cu. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

namespace mamba {

// One decode step over a batch of rows.
struct DecodeArgs {
  int batch, dim, dstate;
  float* state;
  const void* u;
  const void* delta;
  const void* z;
  const void* B;
  const void* C;
  const float* A_log;
  const float* D;
  const float* delta_bias;
  void* out;
  int disc;     // 0 = zero-order hold, 1 = simplified Bbar = dt B
  int* status;  // device status word (see record_status)
  int sms;      // multiprocessors of the device
  unsigned long long wait_ns;  // limit of the bulk kernel's first mbarrier waits (ns); 0 gives up at once
};
cudaError_t launch_state_update(int dtype, const DecodeArgs& a, cudaStream_t stream);

}  // namespace mamba
