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
// 1/A. The register-path kernel takes exp(dt A) - 1 from a four-term series
// when |dt A| < 1/8 (where ex2 - 1 would cancel) and from ex2 - 1 otherwise
// (expm1_acc), so (exp(dt A) - 1) / A keeps a relative error near 1e-6 at any
// dt A; so does the bulk-staged kernel (on B300 the series costs it about 5% at
// N = 16, where its HBM stream is shortest, against ex2 - 1 alone; a per-row
// warp vote between the two cost more). The bulk-staged kernel updates the
// scaled state A h in packed pairs:
// s' = s + (exp(dt A) - 1)(s + B u), h' = s' / A. fp32 inputs use expf /
// expm1f / log1pf. |A| is floored at 1e-20, where exp(dt A) and
// (exp(dt A) - 1) / A equal their A -> 0 limits (1 and dt) in fp32. With the
// simplified discretisation (disc = 1) the input term is dt B u.
#include <algorithm>
#include <type_traits>

#include "device_common.cuh"
#include "decode_args.h"

namespace mamba {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeRows = 4;  // batch rows per thread, loaded together

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
  griddep_launch();
  griddep_wait();

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
      const float A = fminf(PRECISE ? -expf(al) : -hw_ex2(al * kLog2e), -kMinAbsA);
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
            e = expm1_acc(x, ab);
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

// ---------------------------------------------------------------------------
// Bulk-staged decode step for the common layouts (N % 8 == 0, N <= 256,
// dim % 8 == 0, 16-byte aligned pointers). The work is cut into units of one
// batch row of one block of channels. On a 1-D grid (one wave) the units are
// ordered block by block and each CTA walks a contiguous range of them, as
// even as the grid allows, reloading its channels' constants where its range
// enters the next block; on a 2-D grid CTA (x, y) walks rows y, y + gridDim.y,
// ... of block x, so that the CTAs in flight touch neighbouring slabs of the
// same rows. For every unit a 4- or 8-stage ring in shared memory receives,
// by bulk copies that complete on an mbarrier, the row's state slab (8 KB)
// and its u, delta, z, B, C. The threads update the slab in place (8 states
// each), and one thread writes it back with a bulk store. Each thread
// computes A and 1/A for its states once. With an S-stage ring the loads of
// rows i + 1 .. i + S - 1 are in flight while row i is computed, so the kernel
// keeps many bytes in flight without registers.

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

constexpr int kBulkThreads = 256;
constexpr int kBulkFloats = 8;  // states per thread

// Shared-memory layout of one of the S stages (about 8.6 KB each: the slab is
// always 256 / TPC channels x 8 TPC states x 4 bytes = 8 KB): state slab, then
// u, delta, z, B, C.
template <typename Tin, int TPC, int S>
struct BulkGeom {
  static constexpr int kN = TPC * kBulkFloats;  // state size this variant serves
  static constexpr int kCBD = kBulkThreads / TPC;  // channels per block
  static constexpr size_t kState = size_t(kCBD) * kN * 4;
  static constexpr size_t kVec = (size_t(kCBD) * sizeof(Tin) + 15) & ~size_t(15);
  static constexpr size_t kBC = (size_t(kN) * sizeof(Tin) + 15) & ~size_t(15);
  static constexpr size_t kStage = kState + 3 * kVec + 2 * kBC;
  static constexpr size_t kSmem = S * kStage + 8 * S + 128;
};

// Eight consecutive B or C values of one row, from shared memory, as fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// BAL: the 1-D balanced layout (a contiguous range of units per CTA);
// otherwise the 2-D one (rows blockIdx.y, + gridDim.y, ... of block blockIdx.x).
template <typename Tin, int TPC, int DISC, int S, bool BAL>
__global__ void __launch_bounds__(kBulkThreads) state_update_bulk_kernel(const DecodeArgs a) {
  using G = BulkGeom<Tin, TPC, S>;
  using E = Elem<Tin>;
  constexpr bool PRECISE = std::is_same<Tin, float>::value;
  constexpr int N = G::kN, CBD = G::kCBD;
  extern __shared__ unsigned char smem_dyn[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * G::kStage);
  auto st_state = [&](int s) { return reinterpret_cast<float*>(smem + s * G::kStage); };
  auto st_u = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kState); };
  auto st_dl = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kState + G::kVec); };
  auto st_z = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kState + 2 * G::kVec); };
  auto st_B = [&](int s) { return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kState + 3 * G::kVec); };
  auto st_C = [&](int s) {
    return reinterpret_cast<Tin*>(smem + s * G::kStage + G::kState + 3 * G::kVec + G::kBC);
  };

  const int tid = threadIdx.x;
  const int c = tid / TPC, part = tid % TPC;
  const int Dm = a.dim;
  const bool has_z = a.z != nullptr;
  // This CTA's units, walked as (block, row) pairs from (blk0, row0): the
  // next row of the same block, wrapping into the next block (BAL), or rows
  // `step` apart within one block.
  int blk0, row0, nrows, step;
  if constexpr (BAL) {
    const long long units = (long long)((Dm + CBD - 1) / CBD) * a.batch;  // u = block * batch + row
    const long long u0 = units * blockIdx.x / gridDim.x;
    nrows = int(units * (blockIdx.x + 1) / gridDim.x - u0);
    blk0 = int(u0 / a.batch);
    row0 = int(u0 - (long long)blk0 * a.batch);
    step = 1;
  } else {
    blk0 = blockIdx.x;
    row0 = blockIdx.y;
    step = gridDim.y;
    nrows = (a.batch - row0 + step - 1) / step;
  }
  int iss_blk = blk0, iss_row = row0;  // thread 0: the next unit to stage
  // the 2-D layout's one block
  const int nch_fixed = min(CBD, Dm - blk0 * CBD);
  const uint32_t vec_fixed = uint32_t(nch_fixed * sizeof(Tin));
  const uint32_t row_fixed =
      uint32_t(nch_fixed) * N * 4 + (has_z ? 3u : 2u) * vec_fixed + 2u * uint32_t(N * sizeof(Tin));

  auto issue = [&](int i) {  // thread 0: stage unit i of this CTA
    const int s = i % S;
    int b, d0;
    if constexpr (BAL) {  // the unit (iss_blk, iss_row)
      b = iss_row;
      d0 = iss_blk * CBD;
      if (++iss_row == a.batch) {
        iss_row = 0;
        ++iss_blk;
      }
    } else {
      b = row0 + i * step;
      d0 = blk0 * CBD;
    }
    const int nch = BAL ? min(CBD, Dm - d0) : nch_fixed;
    const uint32_t vec_bytes = BAL ? uint32_t(nch * sizeof(Tin)) : vec_fixed;
    const uint32_t row_bytes =
        BAL ? uint32_t(nch) * N * 4 + (has_z ? 3u : 2u) * vec_bytes + 2u * uint32_t(N * sizeof(Tin)) : row_fixed;
    const size_t ch0 = (size_t)b * Dm + d0;
    mbar_arrive_expect_tx(&full[s], row_bytes);
    bulk_load(st_state(s), a.state + ch0 * N, uint32_t(nch) * N * 4, &full[s]);
    bulk_load(st_u(s), static_cast<const Tin*>(a.u) + ch0, vec_bytes, &full[s]);
    bulk_load(st_dl(s), static_cast<const Tin*>(a.delta) + ch0, vec_bytes, &full[s]);
    if (has_z) bulk_load(st_z(s), static_cast<const Tin*>(a.z) + ch0, vec_bytes, &full[s]);
    bulk_load(st_B(s), static_cast<const Tin*>(a.B) + (size_t)b * N, uint32_t(N * sizeof(Tin)), &full[s]);
    bulk_load(st_C(s), static_cast<const Tin*>(a.C) + (size_t)b * N, uint32_t(N * sizeof(Tin)), &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  griddep_launch();
  griddep_wait();
  __syncthreads();
  int issued = 0;  // thread 0
  if (tid == 0)
    for (; issued < min(S - 1, nrows); ++issued) issue(issued);

  // Constants of my channel's 8 states in the current block: A, 1 / A and
  // A log2(e), the last two also as packed pairs for the bf16 path.
  float Av[kBulkFloats], Ik[kBulkFloats];
  float2 A2[kBulkFloats / 2], Al2[kBulkFloats / 2], Ik2[kBulkFloats / 2];
  const int n0 = part * kBulkFloats;
  int blk = -1, d0 = 0, d = 0;
  bool cvalid = false;
  float bias = 0.0f, Dd = 0.0f;
  auto enter_block = [&](int nb) {
    blk = nb;
    d0 = nb * CBD;
    d = d0 + c;
    cvalid = c < min(CBD, Dm - d0);
#pragma unroll
    for (int i = 0; i < kBulkFloats; ++i) {
      const float al = cvalid ? a.A_log[(size_t)d * N + n0 + i] : 0.0f;
      Av[i] = fminf(PRECISE ? -expf(al) : -hw_ex2(al * kLog2e), -kMinAbsA);
      Ik[i] = PRECISE ? 1.0f / Av[i] : hw_rcp(Av[i]);
    }
#pragma unroll
    for (int p = 0; p < kBulkFloats / 2; ++p) {
      A2[p] = make_float2(Av[2 * p], Av[2 * p + 1]);
      Al2[p] = make_float2(Av[2 * p] * kLog2e, Av[2 * p + 1] * kLog2e);
      Ik2[p] = make_float2(Ik[2 * p], Ik[2 * p + 1]);
    }
    bias = (a.delta_bias && cvalid) ? a.delta_bias[d] : 0.0f;
    Dd = (a.D && cvalid) ? a.D[d] : 0.0f;
  };

  if constexpr (!BAL) enter_block(blk0);
  int cur_blk = blk0, b_bal = row0 - 1;  // (BAL) the unit of the iteration below
  for (int i = 0; i < nrows; ++i) {
    const int s = i % S;
    int b;
    if constexpr (BAL) {
      if (++b_bal == a.batch) {
        b_bal = 0;
        ++cur_blk;
      }
      if (cur_blk != blk) enter_block(cur_blk);  // uniform across the CTA
      b = b_bal;
    } else {
      b = row0 + i * step;
    }
    const int nch = BAL ? min(CBD, Dm - d0) : nch_fixed;
    const bool ok = mbar_wait_bounded(&full[s], (i / S) & 1, a.wait_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_status(a.status, kStatusTimeout);
        for (int k = i; k < issued; ++k) mbar_wait_bounded(&full[k % S], (k / S) & 1);
        bulk_wait_all();
      }
      return;
    }
    float* hs = st_state(s) + c * N + n0;
    float y = 0.0f;
    float uf = 0.0f;
    if (cvalid) {
      uf = E::load(st_u(s) + c);
      const float x0 = E::load(st_dl(s) + c) + bias;
      const float dt = PRECISE ? softplus_precise(x0) : softplus_fast(x0);
      float4 h4[2] = {*reinterpret_cast<const float4*>(hs), *reinterpret_cast<const float4*>(hs + 4)};
      float* hv = reinterpret_cast<float*>(h4);
      float Bv[8], Cv[8];
      load8(st_B(s) + n0, Bv);
      load8(st_C(s) + n0, Cv);
      if constexpr (PRECISE) {
#pragma unroll
        for (int k = 0; k < kBulkFloats; ++k) {
          const float e = expm1f(dt * Av[k]);
          const float q = DISC ? dt : ((dt * Av[k] != 0.0f) ? e / Av[k] : dt);  // limit dt as dt A -> 0
          hv[k] = fmaf(e, hv[k], fmaf(q * Bv[k], uf, hv[k]));  // (1 + e) h + q B u
          y = fmaf(Cv[k], hv[k], y);
        }
      } else {
        // bf16: packed pairs. Zero-order hold on the scaled state s = A h:
        // s' = s + (abar - 1)(s + B u), h' = s' / A.
        const float2 dd = make_float2(dt, dt), uu = make_float2(uf, uf);
        float2 yy = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int p = 0; p < kBulkFloats / 2; ++p) {
          const float2 hp = make_float2(hv[2 * p], hv[2 * p + 1]);
          const float2 Bp = make_float2(Bv[2 * p], Bv[2 * p + 1]);
          const float2 x = __fmul2_rn(dd, Al2[p]);
          const float2 ab = make_float2(hw_ex2(x.x), hw_ex2(x.y));
          float2 hn;
          if (DISC == 0) {
            const float2 sp = __fmul2_rn(hp, A2[p]);
            const float2 em1 = make_float2(expm1_acc(x.x, ab.x), expm1_acc(x.y, ab.y));
            hn = __fmul2_rn(__ffma2_rn(em1, __ffma2_rn(Bp, uu, sp), sp), Ik2[p]);
          } else {
            hn = __ffma2_rn(ab, hp, __fmul2_rn(dd, __fmul2_rn(Bp, uu)));  // abar h + dt B u
          }
          yy = __ffma2_rn(make_float2(Cv[2 * p], Cv[2 * p + 1]), hn, yy);
          hv[2 * p] = hn.x;
          hv[2 * p + 1] = hn.y;
        }
        y = yy.x + yy.y;
      }
      *reinterpret_cast<float4*>(hs) = h4[0];
      *reinterpret_cast<float4*>(hs + 4) = h4[1];
    }
#pragma unroll
    for (int off = TPC / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (cvalid && part == 0) {
      y = fmaf(Dd, uf, y);
      if (has_z) {
        const float zf = E::load(st_z(s) + c);
        y *= PRECISE ? silu_precise(zf) : silu_fast(zf);
      }
      E::store(static_cast<Tin*>(a.out) + (size_t)b * Dm + d, y);
    }
    __syncthreads();  // the slab of row i is final in shared memory; stage s is no longer read
    if (tid == 0) {
      fence_proxy_async_smem();
      bulk_store(a.state + ((size_t)b * Dm + d0) * N, st_state(s), uint32_t(nch) * N * 4);
      bulk_commit();
      if (issued < nrows) {
        // the stage of row issued = i + S - 1 held row i - 1, whose store was committed one row ago
        bulk_wait_read_1();
        issue(issued);
        ++issued;
      }
    }
  }
  if (tid == 0) bulk_wait_all();
}

// Whether the bulk-staged path serves these arguments.
template <typename Tin>
static bool decode_bulk_ok(const DecodeArgs& a) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.dstate % 8 == 0 && a.dstate <= 256 && a.dim % 8 == 0 && al16(a.state) && al16(a.u) &&
         al16(a.delta) && (!a.z || al16(a.z)) && al16(a.B) && al16(a.C);
}

// BAL: a 1-D grid of one CTA per slot of every SM at the kernel's occupancy,
// the units dealt out evenly (a CTA walks at most one unit more than
// another); otherwise a 2-D grid of blocks x row groups, about ctas_per_sm
// CTAs per SM.
template <typename Tin, int TPC, int DISC, int S, bool BAL>
static cudaError_t launch_decode_bulk_cfg(const DecodeArgs& a, int ctas_per_sm, cudaStream_t stream) {
  using G = BulkGeom<Tin, TPC, S>;
  static int occupancy = 0;  // per instantiation; benign race (idempotent)
  if (occupancy == 0) {
    cudaError_t e = cudaFuncSetAttribute(state_update_bulk_kernel<Tin, TPC, DISC, S, BAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(G::kSmem));
    int occ = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, state_update_bulk_kernel<Tin, TPC, DISC, S, BAL>,
                                                        kBulkThreads, G::kSmem);
    if (e != cudaSuccess) return e;
    occupancy = std::max(1, occ);
  }
  const int sms = a.sms > 0 ? a.sms : 148;
  const int blocks_x = (a.dim + G::kCBD - 1) / G::kCBD;
  if constexpr (BAL) {
    const long long units = (long long)blocks_x * a.batch;
    const unsigned grid = unsigned(std::max(1LL, std::min(units, (long long)occupancy * sms)));
    return launch_pdl(state_update_bulk_kernel<Tin, TPC, DISC, S, BAL>, dim3(grid), dim3(kBulkThreads), G::kSmem,
                      stream, a);
  }
  const int rb = std::max(1, std::min(a.batch, (ctas_per_sm * sms + blocks_x - 1) / blocks_x));
  return launch_pdl(state_update_bulk_kernel<Tin, TPC, DISC, S, BAL>, dim3(blocks_x, rb), dim3(kBulkThreads),
                    G::kSmem, stream, a);
}

// Ring depth and grid, from sweeps on B300 (batch 128, dim 5120, 2-12 stages,
// 3-32 CTAs per SM):
// - with few channel blocks (small N), exactly one wave of CTAs over balanced
//   ranges of units and a 3-stage ring (N = 16: 17.15 us, against 17.37 us with
//   4 stages, 18.0-20.0 us with 5-8 and 22.2 us with 2; on the earlier 2-D
//   layout one wave beat 2.7 waves of 4-row CTAs, 18.5 against 20.5 us);
// - with many channel blocks (large N), a 5-stage ring over about 11 rows per
//   CTA, 4 CTAs per SM (N = 128: 111.8 us, against 112.3 with
//   6 stages, 112.6 with 4, 127.3 with 8 (3 CTAs per SM) and 157 with 10; 16
//   or 32 CTAs per SM in place of 24: 115.0 and 112.9 us).
template <typename Tin, int TPC, int DISC>
static cudaError_t launch_decode_bulk_disc(const DecodeArgs& a, cudaStream_t stream) {
  const int sms = a.sms > 0 ? a.sms : 148;
  const int blocks_x = (a.dim + BulkGeom<Tin, TPC, 8>::kCBD - 1) / BulkGeom<Tin, TPC, 8>::kCBD;
  if (blocks_x < 2 * sms) return launch_decode_bulk_cfg<Tin, TPC, DISC, 3, true>(a, 0, stream);
  return launch_decode_bulk_cfg<Tin, TPC, DISC, 5, false>(a, 24, stream);
}

template <typename Tin, int TPC>
static cudaError_t launch_decode_bulk(const DecodeArgs& a, cudaStream_t stream) {
  return a.disc == 1 ? launch_decode_bulk_disc<Tin, TPC, 1>(a, stream) : launch_decode_bulk_disc<Tin, TPC, 0>(a, stream);
}

template <typename Tin>
static cudaError_t launch_decode_bulk_typed(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.dstate / 8) {
    case 1: return launch_decode_bulk<Tin, 1>(a, stream);
    case 2: return launch_decode_bulk<Tin, 2>(a, stream);
    case 4: return launch_decode_bulk<Tin, 4>(a, stream);
    case 8: return launch_decode_bulk<Tin, 8>(a, stream);
    case 16: return launch_decode_bulk<Tin, 16>(a, stream);
    case 32: return launch_decode_bulk<Tin, 32>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename Tin, int LPD, int MAXG>
static cudaError_t launch_decode_lpd(const DecodeArgs& a, bool vec, cudaStream_t stream) {
  const int per_block = kDecodeThreads / LPD;
  const dim3 grid(unsigned((a.dim + per_block - 1) / per_block), unsigned((a.batch + kDecodeRows - 1) / kDecodeRows));
  if (vec) return launch_pdl(state_update_kernel<Tin, LPD, MAXG, true>, grid, dim3(kDecodeThreads), 0, stream, a);
  return launch_pdl(state_update_kernel<Tin, LPD, MAXG, false>, grid, dim3(kDecodeThreads), 0, stream, a);
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

// N a power of two from 8 to 256 in the layout the bulk path serves.
static bool bulk_state_size(int n) { return n == 8 || n == 16 || n == 32 || n == 64 || n == 128 || n == 256; }

cudaError_t launch_state_update(int dtype, const DecodeArgs& a, cudaStream_t stream) {
  if (dtype == 0) {
    if (bulk_state_size(a.dstate) && decode_bulk_ok<float>(a)) return launch_decode_bulk_typed<float>(a, stream);
    return launch_decode_typed<float>(a, stream);
  }
  if (bulk_state_size(a.dstate) && decode_bulk_ok<__nv_bfloat16>(a))
    return launch_decode_bulk_typed<__nv_bfloat16>(a, stream);
  return launch_decode_typed<__nv_bfloat16>(a, stream);
}

}  // namespace mamba
