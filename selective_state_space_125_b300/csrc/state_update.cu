// Single-token decode step on a resident fp32 state ("State Space Models and
// Mamba" §3, recurrence mode: one O(1) update of a fixed-size state per token).
//
// Per channel (b, d): dt = softplus(delta + bias_d); for every state n,
//   h_n <- exp(dt A_n) h_n + (exp(dt A_n) - 1) / A_n * B_n u,
//   y    = sum_n C_n h_n + D_d u,  out = y * SiLU(z).
// The step moves 2 * N * 4 bytes of state per channel and reads a few bytes
// of activations, so it is bound by HBM traffic; it therefore always uses the
// accurate expm1f / expf / log1pf forms.
//
// Work layout: LPD threads share a channel; thread i of the group owns states
// 4i .. 4i+3, 4(i + LPD) .. and so on, read and written as one 16-byte vector
// each when N % 4 == 0, so a warp streams 8 * LPD * 16 bytes of contiguous
// state per access. y is reduced across the group with warp shuffles.
#include "device_common.cuh"
#include "scan_args.h"

namespace mamba {

constexpr int kDecodeThreads = 256;

template <typename Tin, int LPD, bool VEC>
__global__ void __launch_bounds__(kDecodeThreads) state_update_kernel(const DecodeArgs a) {
  using E = Elem<Tin>;
  const int g = threadIdx.x % LPD;
  const long long ch = (long long)blockIdx.x * (kDecodeThreads / LPD) + threadIdx.x / LPD;
  const long long nch = (long long)a.batch * a.dim;
  const bool valid = ch < nch;
  const int N = a.dstate;
  const int b = valid ? int(ch / a.dim) : 0;
  const int d = valid ? int(ch % a.dim) : 0;

  float uf = 0.0f, dt = 0.0f;
  if (valid) {
    uf = E::load(static_cast<const Tin*>(a.u) + ch);
    const float x = E::load(static_cast<const Tin*>(a.delta) + ch) + (a.delta_bias ? a.delta_bias[d] : 0.0f);
    dt = softplus_precise(x);
  }
  const Tin* Bb = static_cast<const Tin*>(a.B) + (size_t)b * N;
  const Tin* Cb = static_cast<const Tin*>(a.C) + (size_t)b * N;
  float* hrow = a.state + (size_t)ch * N;
  const float* arow = a.A_log + (size_t)d * N;

  float y = 0.0f;
  for (int n0 = 4 * g; n0 < N; n0 += 4 * LPD) {
    float hv[4], al[4];
    if (valid) {
      if (VEC) {
        const float4 h4 = *reinterpret_cast<const float4*>(hrow + n0);
        const float4 a4 = *reinterpret_cast<const float4*>(arow + n0);
        hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
        al[0] = a4.x; al[1] = a4.y; al[2] = a4.z; al[3] = a4.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hv[i] = (n0 + i < N) ? hrow[n0 + i] : 0.0f;
          al[i] = (n0 + i < N) ? arow[n0 + i] : 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + i;
        if (!VEC && n >= N) break;
        const float A = -expf(al[i]);
        const float x = dt * A;
        const float e = expm1f(x);                           // Abar - 1
        const float coef = (x != 0.0f) ? e / A : dt;         // (Abar - 1) / A, limit dt
        hv[i] = fmaf(coef * E::load(Bb + n), uf, fmaf(e, hv[i], hv[i]));
        y = fmaf(E::load(Cb + n), hv[i], y);
      }
      if (VEC) {
        *reinterpret_cast<float4*>(hrow + n0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < N) hrow[n0 + i] = hv[i];
      }
    }
  }
#pragma unroll
  for (int off = LPD / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
  if (valid && g == 0) {
    y = fmaf(a.D ? a.D[d] : 0.0f, uf, y);
    if (a.z) y *= silu_precise(E::load(static_cast<const Tin*>(a.z) + ch));
    E::store(static_cast<Tin*>(a.out) + ch, y);
  }
}

template <typename Tin, int LPD>
static cudaError_t launch_decode_lpd(const DecodeArgs& a, bool vec, cudaStream_t stream) {
  const long long nch = (long long)a.batch * a.dim;
  const long long per_block = kDecodeThreads / LPD;
  const unsigned grid = unsigned((nch + per_block - 1) / per_block);
  if (vec)
    state_update_kernel<Tin, LPD, true><<<grid, kDecodeThreads, 0, stream>>>(a);
  else
    state_update_kernel<Tin, LPD, false><<<grid, kDecodeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_decode_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int groups = (a.dstate + 3) / 4;  // 4-state groups per channel
  const bool vec = (a.dstate % 4 == 0) && (reinterpret_cast<uintptr_t>(a.state) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.A_log) % 16 == 0);
  if (groups <= 1) return launch_decode_lpd<Tin, 1>(a, vec, stream);
  if (groups <= 2) return launch_decode_lpd<Tin, 2>(a, vec, stream);
  if (groups <= 4) return launch_decode_lpd<Tin, 4>(a, vec, stream);
  if (groups <= 8) return launch_decode_lpd<Tin, 8>(a, vec, stream);
  if (groups <= 16) return launch_decode_lpd<Tin, 16>(a, vec, stream);
  return launch_decode_lpd<Tin, 32>(a, vec, stream);
}

cudaError_t launch_state_update(int dtype, const DecodeArgs& a, cudaStream_t stream) {
  if (dtype == 0) return launch_decode_typed<float>(a, stream);
  return launch_decode_typed<__nv_bfloat16>(a, stream);
}

}  // namespace mamba
