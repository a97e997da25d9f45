// Single-token decode step on a resident fp32 state ("State Space Models and
// Mamba" §3, recurrence mode: one O(1) update of a fixed-size state per token).
//
// Per channel (b, d): dt = softplus(delta + bias_d); for every state n,
//   h_n <- exp(dt A_n) h_n + (exp(dt A_n) - 1) / A_n * B_n u,
//   y    = sum_n C_n h_n + D_d u,  out = y * SiLU(z).
// The step moves 2 * N * 4 bytes of state per channel and reads a few bytes
// of activations, so HBM traffic bounds it once the arithmetic per state is a
// handful of instructions.
//
// Work layout: LPD threads share a channel d; thread i of the group owns
// states 4i .. 4i+3, 4(i + LPD) .. and so on, read and written as one 16-byte
// vector each when N % 4 == 0, so a warp streams 8 * LPD * 16 bytes of
// contiguous state per access. A, 1/A and the per-channel constants are
// computed once per thread and reused for kDecodeRows batch rows, whose loads
// are all issued before any arithmetic. y is reduced across the group with
// warp shuffles.
//
// Math: bf16 inputs use MUFU ex2 for exp(A_log) and exp(dt A) and rcp for
// 1/A; exp(dt A) - 1 comes from a four-term series when |dt A| < 1/8 (where
// ex2 - 1 would cancel) and from ex2 - 1 otherwise, so (exp(dt A) - 1) / A
// keeps a relative error near 1e-6. fp32 inputs use expf / expm1f / log1pf.
// With the simplified discretisation (disc = 1) the input term is dt B u.
#include <type_traits>

#include "device_common.cuh"
#include "scan_args.h"

namespace mamba {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeRows = 4;  // batch rows per thread, loaded together

// exp(x) - 1 for x <= 0 from e = 2^(x log2 e) (a MUFU value of x): series
// below |x| = 1/8 (truncation error < x^5 / 120, relative < 3e-7), e - 1
// above (cancellation error 2^-23 / |x| < 1e-6).
__device__ __forceinline__ float expm1_from_ex2(float x, float e) {
  const float s = x * fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
  return (fabsf(x) < 0.125f) ? s : e - 1.0f;
}

// Four consecutive B or C values of one batch row, loaded in one access and
// widened on use: bf16 keeps the raw 8 bytes (two registers), fp32 a float4.
template <typename T> struct Quad;
template <> struct Quad<__nv_bfloat16> {
  uint2 raw;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { raw = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ void zero() { raw = make_uint2(0u, 0u); }
  __device__ __forceinline__ float get(int i) const {
    const uint32_t w = (i < 2) ? raw.x : raw.y;
    return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};
template <> struct Quad<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void zero() { v = make_float4(0.0f, 0.0f, 0.0f, 0.0f); }
  __device__ __forceinline__ float get(int i) const { return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w)); }
};

// Register budget: 4 CTAs per SM (64 registers) for the vectorised bf16
// path with one 4-state group per thread, 2 otherwise.
template <typename Tin, int MAXG, bool VEC>
struct DecodeMinBlocks {
  static constexpr int value = (VEC && MAXG == 1 && sizeof(Tin) == 2) ? 4 : 2;
};

// MAXG: 4-state groups per thread (1 when LPD covers all groups, i.e.
// N <= 128; 2 for N up to 256 with LPD = 32).
template <typename Tin, int LPD, int MAXG, bool VEC>
__global__ void __launch_bounds__(kDecodeThreads, DecodeMinBlocks<Tin, MAXG, VEC>::value)
    state_update_kernel(const DecodeArgs a) {
  using E = Elem<Tin>;
  constexpr bool PRECISE = std::is_same<Tin, float>::value;
  const int g = threadIdx.x % LPD;
  const int d = blockIdx.x * (kDecodeThreads / LPD) + threadIdx.x / LPD;
  const bool dvalid = d < a.dim;
  const int N = a.dstate;
  const int b0 = blockIdx.y * kDecodeRows;
  const int dd = dvalid ? d : 0;

  // Per-channel constants for my states: Al = A (precise) or A log2(e) (fast), Ik = 1 / A.
  float Al[MAXG][4], Ik[MAXG][4];
  const float* arow = a.A_log + (size_t)dd * N;
#pragma unroll
  for (int k = 0; k < MAXG; ++k) {
    const int n0 = 4 * (g + k * LPD);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = n0 + i;
      const float al = (dvalid && n < N) ? arow[n] : 0.0f;
      const float A = PRECISE ? -expf(al) : -hw_ex2(al * kLog2e);
      Al[k][i] = PRECISE ? A : A * kLog2e;
      Ik[k][i] = PRECISE ? 1.0f / A : hw_rcp(A);
    }
  }
  const float bias = (a.delta_bias && dvalid) ? a.delta_bias[d] : 0.0f;
  const float Dd = (a.D && dvalid) ? a.D[d] : 0.0f;

  // Rows of this CTA that exist (uniform across the CTA).
  const int nrows = min(kDecodeRows, a.batch - b0);

  // Phase 1: issue every load of all rows first (state vectors, token
  // activations, B / C), so that each thread keeps kDecodeRows * MAXG 16-byte
  // state loads in flight instead of one.
  float hv[kDecodeRows][MAXG][4];
  Quad<Tin> Bq[kDecodeRows][MAXG], Cq[kDecodeRows][MAXG];  // used when VEC
  float Bs[VEC ? 1 : kDecodeRows][MAXG][4], Cs[VEC ? 1 : kDecodeRows][MAXG][4];  // otherwise
  float uf[kDecodeRows], xr[kDecodeRows];
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    const int b = b0 + r;
    const bool rv = r < nrows && dvalid;
    const size_t ch = (size_t)(rv ? b : b0) * a.dim + dd;
    uf[r] = rv ? E::load(static_cast<const Tin*>(a.u) + ch) : 0.0f;
    xr[r] = rv ? E::load(static_cast<const Tin*>(a.delta) + ch) : 0.0f;
    const Tin* Bb = static_cast<const Tin*>(a.B) + (size_t)(rv ? b : b0) * N;
    const Tin* Cb = static_cast<const Tin*>(a.C) + (size_t)(rv ? b : b0) * N;
    const float* hrow = a.state + ch * N;
#pragma unroll
    for (int k = 0; k < MAXG; ++k) {
      const int n0 = 4 * (g + k * LPD);
      const bool live = rv && n0 < N;
      if constexpr (VEC) {
        if (live) {
          const float4 h4 = *reinterpret_cast<const float4*>(hrow + n0);
          hv[r][k][0] = h4.x; hv[r][k][1] = h4.y; hv[r][k][2] = h4.z; hv[r][k][3] = h4.w;
          Bq[r][k].load(Bb + n0);
          Cq[r][k].load(Cb + n0);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) hv[r][k][i] = 0.0f;
          Bq[r][k].zero();
          Cq[r][k].zero();
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool in = live && n0 + i < N;
          hv[r][k][i] = in ? hrow[n0 + i] : 0.0f;
          Bs[r][k][i] = in ? E::load(Bb + n0 + i) : 0.0f;
          Cs[r][k][i] = in ? E::load(Cb + n0 + i) : 0.0f;
        }
      }
    }
  }

  // Phase 2: the update and readout of every row, then the stores.
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    const int b = b0 + r;
    const bool rv = r < nrows && dvalid;
    const size_t ch = (size_t)(rv ? b : b0) * a.dim + dd;
    const float x0 = xr[r] + bias;
    const float dt = PRECISE ? softplus_precise(x0) : softplus_fast(x0);
    float* hrow = a.state + ch * N;
    float y = 0.0f;
#pragma unroll
    for (int k = 0; k < MAXG; ++k) {
      const int n0 = 4 * (g + k * LPD);
      const bool live = rv && n0 < N;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = dt * Al[k][i];
        float ab, coef;  // Abar and the factor of B u in Bbar u
        if (a.disc == 1) {
          // simplified discretisation: Bbar = dt B
          ab = PRECISE ? expf(x) : hw_ex2(x);
          coef = dt;
        } else {
          float e;  // Abar - 1
          if (PRECISE) {
            e = expm1f(x);
            ab = 1.0f + e;
          } else {
            ab = hw_ex2(x);
            e = expm1_from_ex2(x * kLn2, ab);
          }
          // (Abar - 1) / A, with the limit dt where dt A underflows to zero
          coef = (x != 0.0f) ? (PRECISE ? e / Al[k][i] : e * Ik[k][i]) : dt;
        }
        const float Bn = VEC ? Bq[r][k].get(i) : Bs[VEC ? 0 : r][k][i];
        const float Cn = VEC ? Cq[r][k].get(i) : Cs[VEC ? 0 : r][k][i];
        hv[r][k][i] = fmaf(coef * Bn, uf[r], ab * hv[r][k][i]);
        y = fmaf(Cn, hv[r][k][i], y);
      }
      if (live) {
        if (VEC) {
          *reinterpret_cast<float4*>(hrow + n0) = make_float4(hv[r][k][0], hv[r][k][1], hv[r][k][2], hv[r][k][3]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (n0 + i < N) hrow[n0 + i] = hv[r][k][i];
        }
      }
    }
#pragma unroll
    for (int off = LPD / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (rv && g == 0) {
      y = fmaf(Dd, uf[r], y);
      if (a.z) {
        const float zf = E::load(static_cast<const Tin*>(a.z) + ch);
        y *= PRECISE ? silu_precise(zf) : silu_fast(zf);
      }
      E::store(static_cast<Tin*>(a.out) + ch, y);
    }
  }
}

template <typename Tin, int LPD, int MAXG>
static cudaError_t launch_decode_lpd(const DecodeArgs& a, bool vec, cudaStream_t stream) {
  const int per_block = kDecodeThreads / LPD;
  const dim3 grid(unsigned((a.dim + per_block - 1) / per_block), unsigned((a.batch + kDecodeRows - 1) / kDecodeRows));
  if (vec)
    state_update_kernel<Tin, LPD, MAXG, true><<<grid, kDecodeThreads, 0, stream>>>(a);
  else
    state_update_kernel<Tin, LPD, MAXG, false><<<grid, kDecodeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_decode_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int groups = (a.dstate + 3) / 4;  // 4-state groups per channel
  const uintptr_t qa = 4 * sizeof(Tin);  // alignment of a 4-element B / C access
  const bool vec = (a.dstate % 4 == 0) && (reinterpret_cast<uintptr_t>(a.state) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.B) % qa == 0) && (reinterpret_cast<uintptr_t>(a.C) % qa == 0);
  if (groups <= 1) return launch_decode_lpd<Tin, 1, 1>(a, vec, stream);
  if (groups <= 2) return launch_decode_lpd<Tin, 2, 1>(a, vec, stream);
  if (groups <= 4) return launch_decode_lpd<Tin, 4, 1>(a, vec, stream);
  if (groups <= 8) return launch_decode_lpd<Tin, 8, 1>(a, vec, stream);
  if (groups <= 16) return launch_decode_lpd<Tin, 16, 1>(a, vec, stream);
  if (groups <= 32) return launch_decode_lpd<Tin, 32, 1>(a, vec, stream);
  return launch_decode_lpd<Tin, 32, 2>(a, vec, stream);
}

cudaError_t launch_state_update(int dtype, const DecodeArgs& a, cudaStream_t stream) {
  if (dtype == 0) return launch_decode_typed<float>(a, stream);
  return launch_decode_typed<__nv_bfloat16>(a, stream);
}

}  // namespace mamba
