// Argument block and launcher of the backward scan, shared by api.cu and
// scan_bwd.cu. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

namespace mamba {

constexpr int kBwdThreads = 128;  // threads per CTA of the backward kernel
constexpr int kBwdChunk = 16;     // time steps per chunk (checkpoint interval)
constexpr int kBwdMaxSegments = 64;
// Smallest |dt A| at which the bf16 backward forms abar - 1 as ex2 - 1
// (relative error below 2^-23 / |dt A| = 2^-9 there), as the forward does.
constexpr float kBwdFastMinDtA = 6.103515625e-05f;  // 2^-14

// Passes of the backward kernel.
constexpr int kBwdFull = 0;    // the gradients over one time segment
constexpr int kBwdFwdAgg = 1;  // a segment's end state from h = 0, and its sum of dt
constexpr int kBwdAdjAgg = 2;  // the adjoint carry a segment passes to its left from a zero carry

struct BwdArgs {
  int batch, dim, dstate, seqlen;
  int nchunk;               // ceil(seqlen / kBwdChunk)
  int nseg;                 // time segments (1 = the whole sequence per CTA)
  int seg_len;              // steps per segment, a multiple of kBwdChunk
  const void* u;            // (B, L, D) input dtype
  const void* delta;
  const void* z;            // or null
  const void* B;            // (B, L, N) input dtype
  const void* C;
  const void* dout;         // (B, L, D) input dtype
  const float* A_log;       // (D, N)
  const float* D;           // (D) or null
  const float* delta_bias;  // (D) or null
  const float* h0;          // (B, D, N) or null
  const float* dlast;       // (B, D, N) or null
  void* du;                 // (B, L, D) input dtype, written
  void* ddelta;
  void* dz;                 // or null
  float* dA_log;            // (D, N), accumulated (zeroed by the caller)
  float* dB;                // (B, L, N), accumulated (zeroed by the caller)
  float* dC;
  float* dD;                // (D) or null, accumulated
  float* ddelta_bias;       // (D) or null, accumulated
  float* dh0;               // (B, D, N) or null, written
  float* ck;                // (B, nchunk, D, N) workspace: the state at each chunk start
  float* seg_h;             // (B, nseg, D, N) workspace: segment end states from h = 0 (segments 0..S-2)
  float* seg_g;             // (B, nseg, D, N) workspace: adjoint carries leaving segments 1..S-1
  float* seg_dsum;          // (B, nseg, D) workspace: sum of dt per segment
  int disc;                 // 0 = zero-order hold, 1 = simplified Bbar = dt B
  int aligned;              // 16-byte vector loads and stores (else element by element)
};

// Whether the backward kernel is built for this state size.
bool scan_bwd_supported(int dstate);
cudaError_t launch_scan_bwd(int dtype, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_scan_bwd_full(int dtype, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_scan_bwd_fwd_agg(int dtype, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_scan_bwd_adj_agg(int dtype, const BwdArgs& a, cudaStream_t stream);

}  // namespace mamba
