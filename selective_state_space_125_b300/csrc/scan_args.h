// Host/device argument blocks of the scan kernels, shared by api.cu and the
// scan translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace mamba {

constexpr int kScanThreads = 128;   // threads per CTA of the scan kernels

struct ScanArgs {
  int batch, dim, dstate, seqlen;
  int nseg;        // time segments run in parallel (1 = whole sequence per CTA)
  int seg_len;     // steps per segment (a multiple of the chunk length)
  const void* u;   // (B, L, D)
  const void* delta;
  const void* z;   // may be null
  const void* B;   // (B, L, N)
  const void* C;
  const float* A_log;       // (D, N)
  const float* D;           // (D) or null
  const float* delta_bias;  // (D) or null
  const float* h0;          // (B, D, N) or null
  void* out;                // (B, L, D)
  float* last_state;        // (B, D, N) or null
  float* agg_h;             // (B, nseg-1, D, N): segment end state started from zero
  float* agg_dsum;          // (B, nseg-1, D): sum of dt over the segment
  int tma_x;                // u/delta/z tiles by TMA (else plain loads)
  int tma_bc;               // B/C tiles by TMA (else plain loads)
  int* status;              // device status word (see record_status)
  const float* conv_w;      // (D, conv_width): fused causal conv1d taps (conv variants only)
  const float* conv_b;      // (D) or null
  int conv_width;           // 1..4
  unsigned long long wait_ns;  // limit of the pipeline's mbarrier waits (ns); 0 gives up at once
  int after_agg;            // full pass launched right after the aggregate pass, with programmatic
                            // stream serialization: it may start early and waits before reading agg_*
};

struct ScanMaps {
  CUtensorMap u, delta, z, B, C;
};

// Geometry of one kernel variant, for the planner.
struct ScanVariant {
  int npl;     // states per thread
  int lpc;     // threads per channel
  int cb;      // channels per CTA
  int chunk;   // time steps per pipeline stage
  size_t smem_bytes;
};

enum class ScanMode { kFull = 0, kAggregate = 1 };

}  // namespace mamba
